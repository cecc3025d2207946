"""kv_copy_blocks (copy on write, page 3 "场景优化1：Parallel Memory Shared")
against the oracle, through the C ABI: bit-exact on whole caches, on the
16-byte path and on the element-by-element path, plus the no-op and
out-of-range cases."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp

from parity import assert_status_ok

pytestmark = pytest.mark.gpu


def _pairs(rng, nb, n):
    """n (src, dst) pairs with distinct destinations that are not sources."""
    perm = rng.permutation(nb)
    dsts = perm[:n]
    srcs = rng.choice(perm[n:], size=n, replace=True)
    return np.stack([srcs, dsts], axis=1).astype(np.int32)


def _random_cache(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    bits = torch.randint(-(1 << 15), 1 << 15, shape, generator=g, device="cuda", dtype=torch.int32)
    return bits.to(torch.int16).view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("shape,npairs", [
    ((2, 3, 40, 16, 2, 64), 9),      # 6 planes, small blocks
    ((2, 4, 24, 256, 8, 128), 7),    # 8 planes of the Qwen3 block shape (512 KiB blocks)
    ((2, 1, 64, 16, 1, 64), 1),      # the tiny configuration's pool, one copy
])
def test_copy_blocks_matches_oracle(shape, npairs):
    rng = np.random.default_rng(hash(shape) & 0xFFFF)
    cache = _random_cache(shape, 7)
    ref = _bits(cache).copy()
    mapping = _pairs(rng, shape[2], npairs)
    kvp.kv_copy_blocks(cache, torch.from_numpy(mapping).cuda())
    torch.cuda.synchronize()
    assert_status_ok()
    oracle.copy_blocks(ref, mapping)
    assert np.array_equal(_bits(cache), ref)


def test_copy_blocks_element_path():
    """block_elems = 12 (not a multiple of 8): the element-by-element kernel."""
    rng = np.random.default_rng(3)
    planes, nb, be = 5, 30, 12
    cache = _random_cache((planes, nb, be), 9)
    ref = _bits(cache).reshape(planes, nb, 1, 1, be).copy()
    mapping = _pairs(rng, nb, 6)
    m = torch.from_numpy(mapping).cuda()
    lib = kvp.library()
    rc = lib.kv_copy_blocks(ctypes.c_void_p(cache.data_ptr()), planes, nb * be, nb, be,
                            ctypes.c_void_p(m.data_ptr()), m.shape[0],
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.kvp_last_error()
    torch.cuda.synchronize()
    assert_status_ok()
    oracle.copy_blocks(ref, mapping)
    assert np.array_equal(_bits(cache).reshape(ref.shape), ref)


def test_copy_blocks_empty_mapping_is_noop():
    cache = _random_cache((2, 2, 8, 16, 1, 64), 1)
    before = _bits(cache).copy()
    kvp.kv_copy_blocks(cache, torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(cache), before)
    assert_status_ok()


def test_copy_blocks_out_of_range_pair_is_skipped_and_flagged():
    cache = _random_cache((2, 2, 8, 16, 1, 64), 2)
    ref = _bits(cache).copy()
    mapping = np.array([[1, 5], [2, 8], [3, 6]], dtype=np.int32)   # pair 1: dst 8 is outside
    kvp.device_status()
    kvp.kv_copy_blocks(cache, torch.from_numpy(mapping).cuda())
    torch.cuda.synchronize()
    assert kvp.device_status() == -6                               # KVP_ERR_DEVICE_DATA
    oracle.copy_blocks(ref, mapping[[0, 2]])
    assert np.array_equal(_bits(cache), ref)


def test_copy_then_store_then_attend_parallel_sampling():
    """The pages' copy-on-write flow on the GPU: two sequences share a partly
    filled block; A1 gets a copy, both append a token, and decode attention
    over each sequence equals the oracle's."""
    from paged_kv_cache_125_gb300 import workloads as W
    from parity import assert_attn_close
    g = torch.Generator().manual_seed(4)
    nb, bs, hkv, d, hq = 16, 16, 2, 64, 4
    kv = torch.full((2, 1, nb, bs, hkv, d), float("nan"), dtype=torch.bfloat16)
    prompt_len = 21
    table = [11, 3]
    pk = torch.randn((prompt_len, hkv, d), generator=g).to(torch.bfloat16)
    pv = torch.randn((prompt_len, hkv, d), generator=g).to(torch.bfloat16)
    kvc = kv.cuda()
    slots = torch.tensor(W.slots_of_positions(table, range(prompt_len), bs), dtype=torch.int32)
    kvp.kv_store(pk.cuda(), pv.cuda(), slots.cuda(), kvc[0, 0], kvc[1, 0])
    kvp.kv_copy_blocks(kvc, torch.tensor([[3, 9]], dtype=torch.int32, device="cuda"))
    tables = [[11, 9], [11, 3]]
    nk = torch.randn((2, hkv, d), generator=g).to(torch.bfloat16)
    nv = torch.randn((2, hkv, d), generator=g).to(torch.bfloat16)
    s2 = torch.tensor([W.slots_of_positions(t, [prompt_len], bs)[0] for t in tables], dtype=torch.int32)
    kvp.kv_store(nk.cuda(), nv.cuda(), s2.cuda(), kvc[0, 0], kvc[1, 0])
    q = torch.randn((2, hq, d), generator=g).to(torch.bfloat16)
    bt = torch.tensor(tables, dtype=torch.int32)
    ctx = torch.tensor([prompt_len + 1] * 2, dtype=torch.int32)
    out = kvp.attn_decode_paged(q.cuda(), kvc[0, 0], kvc[1, 0], bt.cuda(), ctx.cuda(), prompt_len + 1,
                                softmax_scale=d ** -0.5)
    torch.cuda.synchronize()
    assert_status_ok()
    kr = kv[0, 0].view(torch.int16).numpy().view(np.uint16).copy()
    vr = kv[1, 0].view(torch.int16).numpy().view(np.uint16).copy()
    oracle.kv_store(pk, pv, slots, kr, vr)
    both = np.stack([kr, vr])[:, None]
    oracle.copy_blocks(both, [[3, 9]])
    kr, vr = np.ascontiguousarray(both[0, 0]), np.ascontiguousarray(both[1, 0])
    oracle.kv_store(nk, nv, s2, kr, vr)
    ref = oracle.decode(q, kr, vr, bt, ctx, hq, hkv, d ** -0.5)
    assert_attn_close(out, ref, "copy-on-write decode")
