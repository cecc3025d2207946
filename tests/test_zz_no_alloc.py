"""attn_decode_paged_noalloc, the decode entry point for callers that cannot
allocate device memory (it uses the library's built-in scratch instead of a
caller workspace).  Called through the C ABI and checked against the fp64
oracle and against attn_decode_paged.  Two calls in a row use the same number
of CTAs with other lengths and values, so the second call would read what the
first one left in the shared scratch if any partial it merges were stale; a
third call uses fewer CTAs.  This file is collected last on purpose."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

from parity import MAX_ABS, MEAN_ABS, assert_attn_close, gpu_pool, u16

pytestmark = pytest.mark.gpu


def _raw_noalloc(q, kc, vc, bt, ctx, max_ctx, scale, out):
    lib = kvp.library()
    nb, bs, hkv, d = kc.shape
    b, hq, _ = q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.attn_decode_paged_noalloc(
        ctypes.c_void_p(q.data_ptr()), q.stride(0), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()), nb, bs, ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
        ctypes.c_void_p(ctx.data_ptr()), b, max_ctx, hq, hkv, d, scale,
        ctypes.c_void_p(out.data_ptr()), out.stride(0), stream)


def _case(w, negate_q=False):
    kc, vc = gpu_pool(w)
    st = w.steps[0].store
    kvp.kv_store(st.k.cuda(), st.v.cuda(), st.slot_mapping.cuda(), kc, vc)
    a = w.steps[0].attn
    m = a.meta
    q = (-a.q if negate_q else a.q).cuda()
    return kc, vc, q, m.block_tables.cuda(), m.context_lens.cuda(), m.max_context_len


def test_noalloc_matches_oracle_and_workspace_entry_point_on_calls_in_a_row():
    lens_a = [1000, 37, 4096, 513, 1]
    cases = [
        (W.decode_workload("noalloc_a", lens_a, 32, 8, 128, 64, 128), False),
        # same num_seqs and max_context_len (same CTA count), other cut points and values
        (W.decode_workload("noalloc_a2", [4096, 1, 513, 37, 1000], 32, 8, 128, 64, 128), True),
        (W.decode_workload("noalloc_b", [300, 17, 64, 2000], 16, 8, 128, 16, 256), False),
    ]
    runs = []
    for w, neg in cases:  # the no-alloc calls back to back on one stream
        kc, vc, q, bt, ctx, max_ctx = _case(w, neg)
        scale = 1.0 / math.sqrt(w.head_dim)
        out = torch.full_like(q, float("nan"))
        rc = _raw_noalloc(q, kc, vc, bt, ctx, max_ctx, scale, out)
        assert rc == 0, kvp.library().kvp_last_error()
        runs.append((w, kc, vc, q, bt, ctx, max_ctx, scale, out))
    torch.cuda.synchronize()
    assert kvp.device_status() == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # the decode plan: one CTA per 64 tokens of num_seqs x max_context_len, at most one per SM
    ctas = [min(sms, -(-len(r[5]) * r[6] // 64)) for r in runs]
    assert ctas[0] == ctas[1] and ctas[2] < ctas[0], ctas
    for w, kc, vc, q, bt, ctx, max_ctx, scale, out in runs:
        m = w.steps[0].attn.meta
        ref = oracle.decode(q.cpu(), u16(kc), u16(vc), m.block_tables, m.context_lens, w.num_heads,
                            w.num_kv_heads, scale)
        assert_attn_close(out, ref, f"{w.name} against the oracle")
        other = kvp.attn_decode_paged(q, kc, vc, bt, ctx, max_ctx, softmax_scale=scale)
        g, r = out.float().cpu().numpy(), other.float().cpu().numpy()
        err = np.abs(g - r)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (w.name, err.max(), err.mean())


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """64 query heads at head_dim 128 need more partial space than 8 MiB once
    the batch spreads over more than 124 CTAs; the scratch check comes after
    the argument checks of attn_decode_paged."""
    kc = torch.zeros((4, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    ctx = torch.ones(1, dtype=torch.int32, device="cuda")
    need = kvp.attn_decode_workspace_size(1, 64, 128, 1 << 20, 16)
    if need <= (8 << 20):
        pytest.skip("this device's SM count keeps the shape inside the scratch")
    rc = _raw_noalloc(q, kc, kc.clone(), bt, ctx, 1 << 20, 0.125, torch.empty_like(q))
    assert rc == -3
    assert b"built-in scratch" in kvp.library().kvp_last_error()
    # an unsupported shape is reported as attn_decode_paged reports it
    rc = _raw_noalloc(torch.zeros((1, 24, 128), dtype=torch.bfloat16, device="cuda"), kc, kc, bt, ctx,
                      1 << 20, 0.125, torch.empty((1, 24, 128), dtype=torch.bfloat16, device="cuda"))
    assert rc == -2 and b"attn_decode_paged_noalloc: unsupported heads" in kvp.library().kvp_last_error()
