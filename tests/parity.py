"""Runs a seeded workload through the CUDA library and through the CPU oracle
and compares them.  Test infrastructure (imports the oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

# Attention outputs: bf16 results vs the fp64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
BF16_NAN = 0x7FC0


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_pool(w: W.Workload):
    shape = w.cache_shape()
    kc = np.full(shape, BF16_NAN, np.uint16)
    vc = np.full(shape, BF16_NAN, np.uint16)
    if w.history_slots is not None:
        idx = w.history_slots.numpy()
        kc.reshape(-1, w.num_kv_heads, w.head_dim)[idx] = u16(w.history_k)
        vc.reshape(-1, w.num_kv_heads, w.head_dim)[idx] = u16(w.history_v)
    return kc, vc


def run_oracle(w: W.Workload, rows_for=None, seqs_for=None):
    """-> (per-step fp64 outputs, k_cache, v_cache) as numpy."""
    kc, vc = oracle_pool(w)
    for st in w.setup:
        oracle.kv_store(st.k, st.v, st.slot_mapping, kc, vc)
    outs = []
    for i, step in enumerate(w.steps):
        oracle.kv_store(step.store.k, step.store.v, step.store.slot_mapping, kc, vc)
        a = step.attn
        if step.is_prefill:
            m = a.meta
            rows = rows_for(i) if rows_for else None
            if m.block_tables is not None:
                o = oracle.prefill(a.q, m.cu_seqlens_q, m.cu_seqlens_k, w.num_heads, w.num_kv_heads,
                                   w.scale, k_cache=kc, v_cache=vc, block_tables=m.block_tables, rows=rows)
            else:
                o = oracle.prefill(a.q, m.cu_seqlens_q, m.cu_seqlens_k, w.num_heads, w.num_kv_heads,
                                   w.scale, k=a.k, v=a.v, rows=rows)
        else:
            m = a.meta
            seqs = seqs_for(i) if seqs_for else None
            o = oracle.decode(a.q, kc, vc, m.block_tables, m.context_lens, w.num_heads,
                              w.num_kv_heads, w.scale, seqs=seqs)
        outs.append(o)
    return outs, kc, vc


def gpu_pool(w: W.Workload, device="cuda"):
    kc, vc = w.new_cache(device, poison=True)
    w.place_history(kc, vc)
    return kc, vc


def run_gpu(w: W.Workload, device="cuda", fused_decode=False, fused_prefill=False):
    """-> (per-step bf16 outputs on the device, k_cache, v_cache).  With
    fused_decode, decode steps go through attn_decode_paged_append (store and
    attention in one launch) instead of kv_store + attn_decode_paged; with
    fused_prefill, prefill steps through attn_prefill_varlen_append."""
    kc, vc = gpu_pool(w, device)
    for st in w.setup:
        kvp.kv_store(st.k.to(device), st.v.to(device), st.slot_mapping.to(device), kc, vc)
    outs = []
    for step in w.steps:
        s = step.store
        a = step.attn
        m = a.meta
        if fused_decode and not step.is_prefill:
            outs.append(kvp.attn_decode_paged_append(
                a.q.to(device), s.k.to(device), s.v.to(device), s.slot_mapping.to(device), kc, vc,
                m.block_tables.to(device), m.context_lens.to(device), m.max_context_len,
                softmax_scale=w.scale))
            continue
        if fused_prefill and step.is_prefill:
            bt = None if m.block_tables is None else m.block_tables.to(device)
            outs.append(kvp.attn_prefill_varlen_append(
                a.q.to(device), s.k.to(device), s.v.to(device), s.slot_mapping.to(device),
                m.cu_seqlens_q.to(device), m.cu_seqlens_k.to(device), m.max_seqlen_q, m.max_seqlen_k,
                kc, vc, block_tables=bt, softmax_scale=w.scale))
            continue
        kvp.kv_store(s.k.to(device), s.v.to(device), s.slot_mapping.to(device), kc, vc)
        if step.is_prefill:
            bt = None if m.block_tables is None else m.block_tables.to(device)
            o = kvp.attn_prefill_varlen(a.q.to(device), m.cu_seqlens_q.to(device), m.cu_seqlens_k.to(device),
                                        m.max_seqlen_q, m.max_seqlen_k, k=a.k.to(device), v=a.v.to(device),
                                        k_cache=kc, v_cache=vc, block_tables=bt,
                                        num_kv_heads=w.num_kv_heads, softmax_scale=w.scale)
        else:
            o = kvp.attn_decode_paged(a.q.to(device), kc, vc, m.block_tables.to(device),
                                      m.context_lens.to(device), m.max_context_len, softmax_scale=w.scale)
        outs.append(o)
    torch.cuda.synchronize()
    return outs, kc, vc


def assert_attn_close(gpu: torch.Tensor, ref: np.ndarray, what: str, mask=None):
    g = gpu.detach().float().cpu().double().numpy()
    if mask is not None:
        g, ref = g[mask], ref[mask]
    assert np.isfinite(g).all(), f"{what}: non-finite values in the CUDA output"
    err = np.abs(g - ref)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max-abs {mx:.3e}, mean-abs {mean:.3e}"
    return mx, mean


def assert_status_ok():
    st = kvp.device_status()
    assert st == 0, f"device status {st} ({kvp.ERROR_NAMES.get(st)})"
