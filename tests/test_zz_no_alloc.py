"""attn_decode_paged_noalloc, the decode entry point for callers that cannot
allocate device memory (it uses the library's built-in scratch instead of a
caller workspace).  Called through the C ABI and checked against
attn_decode_paged on two calls in a row with different batches, so the second
call also shows that nothing left in the shared scratch by the first one leaks
into its result.  This file is collected last on purpose."""
import ctypes
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

from parity import MAX_ABS, MEAN_ABS, gpu_pool

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


def _case(w):
    kc, vc = gpu_pool(w)
    st = w.steps[0].store
    kvp.kv_store(st.k.cuda(), st.v.cuda(), st.slot_mapping.cuda(), kc, vc)
    a = w.steps[0].attn
    m = a.meta
    q, bt, ctx = a.q.cuda(), m.block_tables.cuda(), m.context_lens.cuda()
    return kc, vc, q, bt, ctx, m.max_context_len


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [W.decode_workload("noalloc_a", [1000, 37, 4096, 513, 1], 32, 8, 128, 256, 64),
             W.decode_workload("noalloc_b", [300, 17, 64, 2000], 16, 8, 128, 16, 256)]
    for w in cases:
        kc, vc, q, bt, ctx, max_ctx = _case(w)
        scale = 1.0 / math.sqrt(w.head_dim)
        ref = kvp.attn_decode_paged(q, kc, vc, bt, ctx, max_ctx, softmax_scale=scale)
        out = torch.full_like(q, float("nan"))
        rc = _raw_noalloc(q, kc, vc, bt, ctx, max_ctx, scale, out)
        assert rc == 0, kvp.library().kvp_last_error()
        torch.cuda.synchronize()
        assert kvp.device_status() == 0
        g = out.float().cpu().numpy()
        r = ref.float().cpu().numpy()
        assert np.isfinite(g).all()
        err = np.abs(g - r)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (w.name, err.max(), err.mean())


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """64 query heads at head_dim 128 need more partial space than 8 MiB on a
    152-SM GPU; the size check comes before anything else."""
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
