"""GPU parity: kv_store (bit-exact) and attn_decode_paged (fp tolerance) against
the CPU oracle, through the C ABI, on seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

from parity import (BF16_NAN, assert_attn_close, assert_status_ok, gpu_pool, oracle_pool, run_gpu,
                    run_oracle, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    kvp.device_status()
    yield
    assert_status_ok()


# --------------------------------------------------------------------------- kv_store

def _random_store_case(seed, n, nb, bs, hkv, d, pad_every=0):
    g = torch.Generator().manual_seed(seed)
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int32)
    if pad_every:
        slots[::pad_every] = -1
    k = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16)
    return k, v, slots


@pytest.mark.parametrize("n,nb,bs,hkv,d,pad", [(1, 4, 16, 1, 64, 0), (301, 64, 16, 1, 64, 7),
                                               (4096, 256, 256, 8, 128, 0), (777, 100, 32, 2, 128, 5),
                                               (50, 8, 16, 3, 36, 4)])
def test_kv_store_bit_exact(n, nb, bs, hkv, d, pad):
    k, v, slots = _random_store_case(n + d, n, nb, bs, hkv, d, pad)
    kc_ref = np.full((nb, bs, hkv, d), BF16_NAN, np.uint16)
    vc_ref = kc_ref.copy()
    oracle.kv_store(k, v, slots, kc_ref, vc_ref)
    kc = torch.full((nb, bs, hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    kvp.kv_store(k.cuda(), v.cuda(), slots.cuda(), kc, vc)
    assert np.array_equal(u16(kc), kc_ref) and np.array_equal(u16(vc), vc_ref)


def test_kv_store_strided_rows_from_fused_qkv():
    """k and v as column slices of one fused [N, (Hq + 2 Hkv) * d] projection."""
    n, hq, hkv, d, nb, bs = 200, 4, 2, 128, 32, 16
    g = torch.Generator().manual_seed(3)
    qkv = torch.randn((n, (hq + 2 * hkv) * d), generator=g).to(torch.bfloat16).cuda()
    k = qkv[:, hq * d:(hq + hkv) * d].view(n, hkv, d)
    v = qkv[:, (hq + hkv) * d:].view(n, hkv, d)
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int32)
    kc = torch.full((nb, bs, hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    kvp.kv_store(k, v, slots.cuda(), kc, vc)
    kr = np.full((nb, bs, hkv, d), BF16_NAN, np.uint16)
    vr = kr.copy()
    oracle.kv_store(k.cpu().contiguous(), v.cpu().contiguous(), slots, kr, vr)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)


def test_kv_store_empty_is_noop():
    kc = torch.zeros((2, 16, 1, 64), dtype=torch.bfloat16, device="cuda")
    e = torch.empty((0, 1, 64), dtype=torch.bfloat16, device="cuda")
    kvp.kv_store(e, e, torch.empty(0, dtype=torch.int32, device="cuda"), kc, kc.clone())
    assert kc.abs().sum().item() == 0


def test_kv_store_out_of_range_slot_is_skipped_and_flagged():
    kc = torch.zeros((2, 16, 1, 64), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    k = torch.ones((2, 1, 64), dtype=torch.bfloat16, device="cuda")
    kvp.kv_store(k, k, torch.tensor([32, 3], dtype=torch.int32, device="cuda"), kc, vc)
    assert kvp.device_status() == -6  # KVP_ERR_DEVICE_DATA
    assert kc.view(32, 64)[3].eq(1).all() and kc.view(32, 64).sum().item() == 64


# --------------------------------------------------------------------------- decode

def _check_decode_workload(w, seqs=None, fused=False):
    outs, kc, vc = run_gpu(w, fused_decode=fused)
    ref, kr, vr = run_oracle(w, seqs_for=(lambda i: seqs) if seqs is not None else None)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr), "cache differs after kv_store"
    mask = None if seqs is None else np.asarray(seqs)
    return assert_attn_close(outs[0], ref[0], w.name, mask)


def test_decode_config2_full_size():
    """64 sequences, Qwen3-0.6B heads (16/8/128), context U[512, 4096], bs 256."""
    _check_decode_workload(W.config2_decode())


@pytest.mark.parametrize("hq,hkv,d,bs,lens", [
    (2, 1, 64, 16, [1, 16, 17, 300, 33]),
    (8, 8, 128, 256, [5000, 1, 256, 257, 700]),
    (16, 8, 128, 16, [3, 40, 129, 1024]),
    (32, 8, 128, 256, [8192, 128, 4096]),
    (4, 4, 64, 32, [999, 64]),
    (4, 2, 128, 48, [47, 48, 49, 2000]),
    (8, 2, 64, 16, [300, 301]),
    (8, 1, 64, 64, [1000]),
    (4, 1, 128, 16, [70, 15]),
    (64, 8, 128, 256, [3000, 1, 255, 257]),                      # G=8 at head_dim 128
    (16, 2, 128, 32, [700, 33]),
])
def test_decode_shapes_and_ragged_lengths(hq, hkv, d, bs, lens):
    nb = sum(W.num_blocks_for(L, bs) for L in lens) + 7
    w = W.decode_workload(f"decode_{hq}_{hkv}_{d}_{bs}", lens, hq, hkv, d, bs, nb)
    _check_decode_workload(w)


def test_decode_single_long_sequence_crosses_every_cta():
    """One sequence spread over all CTAs: every CTA leaves a partial and the
    log-sum-exp merge combines them."""
    w = W.decode_workload("long", [65536], 16, 8, 128, 256, 300)
    _check_decode_workload(w)


def test_decode_zero_context_rows_are_zero():
    w = W.decode_workload("with_padding", [100, 1, 700], 4, 2, 128, 16, 64)
    step = w.steps[0]
    kc, vc = gpu_pool(w)
    m = step.attn.meta
    ctx = m.context_lens.clone()
    ctx[1] = 0  # a padded row of a CUDA-graph batch
    out = kvp.attn_decode_paged(step.attn.q.cuda(), kc, vc, m.block_tables.cuda(), ctx.cuda(),
                                m.max_context_len, softmax_scale=w.scale)
    assert out[1].float().abs().max().item() == 0.0
    kr, vr = oracle_pool(w)
    ref = oracle.decode(step.attn.q, kr, vr, m.block_tables, ctx, 4, 2, w.scale)
    # rows 0 and 2 still read their history (the new token was never stored -> NaN-free slots only)
    ctx2 = ctx.clone()
    ctx2[0] -= 1
    ctx2[2] -= 1
    out2 = kvp.attn_decode_paged(step.attn.q.cuda(), kc, vc, m.block_tables.cuda(), ctx2.cuda(),
                                 m.max_context_len, softmax_scale=w.scale)
    ref2 = oracle.decode(step.attn.q, kr, vr, m.block_tables, ctx2, 4, 2, w.scale)
    assert_attn_close(out2, ref2, "padding rows")
    assert np.all(ref[1] == 0)


def test_decode_all_rows_empty():
    kc = torch.full((4, 16, 2, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    q = torch.randn((3, 4, 64), device="cuda").to(torch.bfloat16)
    bt = torch.full((3, 2), -1, dtype=torch.int32, device="cuda")
    out = kvp.attn_decode_paged(q, kc, kc.clone(), bt, torch.zeros(3, dtype=torch.int32, device="cuda"), 0)
    assert out.float().abs().max().item() == 0.0


def test_decode_out_of_range_block_is_flagged_not_read():
    w = W.decode_workload("bad_block", [40, 40], 4, 2, 64, 16, 16)
    kc, vc = gpu_pool(w)
    m = w.steps[0].attn.meta
    bt = m.block_tables.clone()
    bt[1, 1] = 10_000
    kvp.attn_decode_paged(w.steps[0].attn.q.cuda(), kc, vc, bt.cuda(), m.context_lens.cuda(),
                          m.max_context_len)
    assert kvp.device_status() == -6


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_store"])
def test_decode_config4_full_pool_all_sequences(fused):
    """512 sequences, Qwen3-8B heads, ~150 GB pool: every sequence's output
    against the oracle and the stored slots bit-exact, through kv_store +
    attn_decode_paged and through attn_decode_paged_append (the call the
    benchmark times).  The oracle reads a compact host copy of the blocks the
    sequences reference, 64 sequences at a time (about 7 GB of K/V in all)."""
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < 170e9:
        pytest.skip("needs ~160 GB of free device memory")
    w = W.config4_decode(device="cuda")
    outs, kc, vc = run_gpu(w, fused_decode=fused)
    m = w.steps[0].attn.meta
    # stored K/V of this step, bit-exact
    st = w.steps[0].store
    flat_k, flat_v = kc.view(-1, 8, 128), vc.view(-1, 8, 128)
    idx = st.slot_mapping.long().cuda()
    assert torch.equal(flat_k[idx].view(torch.int16), st.k.view(torch.int16))
    assert torch.equal(flat_v[idx].view(torch.int16), st.v.view(torch.int16))
    out_host = outs[0].cpu()
    q_host = w.steps[0].attn.q.cpu()
    for c0 in range(0, 512, 64):
        seqs = list(range(c0, c0 + 64))
        tables, ctxs, blocks = [], [], []
        for b in seqs:
            L = int(m.context_lens[b])
            row = m.block_tables[b, :W.num_blocks_for(L, 256)].tolist()
            tables.append(list(range(len(blocks), len(blocks) + len(row))))
            blocks += row
            ctxs.append(L)
        bidx = torch.tensor(blocks, dtype=torch.long, device="cuda")
        kh, vh = u16(kc[bidx]), u16(vc[bidx])
        ref = oracle.decode(q_host[seqs], kh, vh, W.prepare_block_tables(tables),
                            torch.tensor(ctxs, dtype=torch.int32), 32, 8, w.scale)
        assert_attn_close(out_host[seqs], ref, f"config4 sequences {c0}..{c0 + 63}")
        del kh, vh
    del outs, kc, vc
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- fused store + decode

def test_decode_append_config2_full_size():
    """attn_decode_paged_append on the 64-sequence step: the cache after the
    call is bit-exact (store), the outputs match the oracle's store-then-decode."""
    _check_decode_workload(W.config2_decode(), fused=True)


@pytest.mark.parametrize("hq,hkv,d,bs,lens", [
    (2, 1, 64, 16, [1, 16, 17, 300, 33]),
    (8, 8, 128, 256, [5000, 1, 256, 257, 700]),
    (32, 8, 128, 256, [8192, 128, 4096]),
    (4, 2, 128, 48, [47, 48, 49, 2000]),
    (8, 1, 64, 64, [1000]),
    (64, 8, 128, 256, [3000, 1, 255, 257]),
])
def test_decode_append_shapes_and_ragged_lengths(hq, hkv, d, bs, lens):
    """New rows at the first slot of a block (stage of one token), mid-block and
    at a block's last slot; group sizes 1..8."""
    nb = sum(W.num_blocks_for(L, bs) for L in lens) + 7
    w = W.decode_workload(f"append_{hq}_{hkv}_{d}_{bs}", lens, hq, hkv, d, bs, nb)
    _check_decode_workload(w, fused=True)


def test_decode_append_long_sequence_crosses_every_cta():
    """The new token lands in the last CTA's chunk of a sequence split over all
    CTAs; the others read only stored history."""
    w = W.decode_workload("append_long", [65536, 3], 16, 8, 128, 256, 300)
    _check_decode_workload(w, fused=True)


def test_decode_append_padding_rows():
    """Rows with slot -1 and context 0 (the graph path's padding) store nothing
    and produce zeros; the other rows are unaffected."""
    w = W.decode_workload("append_pad", [100, 1, 700], 4, 2, 128, 16, 64)
    step = w.steps[0]
    kc, vc = gpu_pool(w)
    m, st = step.attn.meta, step.store
    ctx, slots = m.context_lens.clone(), st.slot_mapping.clone()
    ctx[1], slots[1] = 0, -1
    before = u16(kc).copy()
    out = kvp.attn_decode_paged_append(step.attn.q.cuda(), st.k.cuda(), st.v.cuda(), slots.cuda(), kc,
                                       vc, m.block_tables.cuda(), ctx.cuda(), m.max_context_len,
                                       softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert out[1].float().abs().max().item() == 0.0
    kr, vr = oracle_pool(w)
    oracle.kv_store(st.k, st.v, slots, kr, vr)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    changed = np.argwhere((u16(kc) != before).any(axis=(2, 3)))
    assert len(changed) == 2  # the two stored rows only
    ref = oracle.decode(step.attn.q, kr, vr, m.block_tables, ctx, 4, 2, w.scale)
    assert_attn_close(out, ref, "append with padding rows")


def test_decode_append_slot_mismatch_is_flagged():
    """A slot that is not the one of position context_len - 1 is reported
    (KVP_ERR_DEVICE_DATA); the row is still stored there."""
    w = W.decode_workload("append_bad_slot", [40, 40], 4, 2, 64, 16, 16)
    step = w.steps[0]
    kc, vc = gpu_pool(w)
    m, st = step.attn.meta, step.store
    slots = st.slot_mapping.clone()
    slots[0] = int(slots[0]) - 1  # an earlier slot of the same block
    kvp.attn_decode_paged_append(step.attn.q.cuda(), st.k.cuda(), st.v.cuda(), slots.cuda(), kc, vc,
                                 m.block_tables.cuda(), m.context_lens.cuda(), m.max_context_len)
    assert kvp.device_status() == -6
    flat = kc.view(-1, 2, 64)
    assert torch.equal(flat[int(slots[0])].cpu().view(torch.int16), st.k[0].view(torch.int16))
