"""GPU parity of attn_prefill_varlen_append, the prefill step of one layer in
one launch: the store of the step's new rows fused into the varlen prefill
("nano-vLLM-1" "4. prefill 输入打包": slot_mapping holds the slots of the
uncached tokens, one per query row, and the keys of a prefix hit are read
through block_tables).  Its result must equal kv_store followed by
attn_prefill_varlen for any metadata: the caches bit-exact against the
oracle's store, the outputs against the oracle's prefill."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

from parity import (assert_attn_close, assert_status_ok, gpu_pool, oracle_pool, run_gpu, run_oracle,
                    u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    kvp.device_status()
    yield


def _check(w, rows_for=None):
    outs, kc, vc = run_gpu(w, fused_prefill=True)
    assert_status_ok()
    ref, kr, vr = run_oracle(w, rows_for=rows_for)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr), "caches differ after the store"
    for i, (o, r) in enumerate(zip(outs, ref)):
        mask = None if rows_for is None or not w.steps[i].is_prefill else rows_for(i)
        assert_attn_close(o, r, f"{w.name} step {i}", mask)


def test_append_config3_full_size():
    """The prefill configuration: 8 prompts U[256, 2048], 0-2 cached blocks,
    Qwen3-8B heads, bs 256; every row."""
    _check(W.config3_prefill())


def test_append_tiny_pipeline():
    _check(W.config1_tiny())


@pytest.mark.parametrize("hq,hkv,d,bs,lens,cached", [
    (2, 2, 64, 16, [1, 2, 129, 300], [0, 0, 0, 0]),            # packed (no prefix), G=1
    (4, 2, 128, 16, [45, 200, 333], [1, 0, 4]),                  # paged, bs 16
    (8, 2, 128, 32, [640, 70], [5, 2]),
    (16, 2, 64, 256, [1000, 257, 256], [1, 0, 0]),               # G=8, d 64
    (32, 8, 128, 256, [2048, 1, 130], [7, 0, 0]),
    (16, 8, 128, 128, [777, 128, 129], [2, 0, 1]),
    (8, 8, 128, 64, [300, 301, 302, 303, 304], [0, 1, 2, 3, 4]),
    (16, 8, 128, 256, [100, 900, 2000, 37], [0, 0, 0, 0]),       # packed, several kv tiles
    (16, 8, 128, 256, [16384], [0]),                             # one long prompt: every CTA stores
])
def test_append_shapes(hq, hkv, d, bs, lens, cached):
    nb = sum(W.num_blocks_for(L, bs) for L in lens) + 5
    _check(W.prefill_workload(f"pfa_{hq}_{hkv}_{d}_{bs}", lens, cached, hq, hkv, d, bs, nb))


def test_append_prefix_written_in_the_same_call():
    """Sequence 1's cached prefix is sequence 0's first two blocks, which this
    very call stores (two requests with the same prompt prefix scheduled in
    one prefill step): the store must land before any key tile is loaded."""
    hq, hkv, d, bs = 16, 8, 128, 256
    A, B, C, D = 3, 7, 1, 5
    lens, cached, tables = [600, 700, 530], [0, 512, 512], [[A, B, C], [A, B, D], [A, B, 2]]
    meta = W.prefill_metadata(lens, cached, tables, bs)
    tq = int(meta.cu_seqlens_q[-1])
    g = W.generator(W.SEED_VALUES)
    q = W.randn_bf16((tq, hq, d), g)
    k = W.randn_bf16((tq, hkv, d), g)
    v = W.randn_bf16((tq, hkv, d), g)
    w = W.Workload("same_call_prefix", hq, hkv, d, bs, 8,
                   [W.Step(W.StoreCall(k, v, meta.slot_mapping), W.PrefillCall(q, k, v, meta))])
    assert meta.block_tables is not None
    _check(w)


def test_append_mixed_step_full_size_sampled():
    """The bench's mixed step (4 prefill chunks + 128 decode rows, 32/8/128)
    through the fused call; every decode row and every 5th chunk row."""
    w = W.mixed_step_workload()
    m = w.steps[0].attn.meta
    cu = m.cu_seqlens_q.tolist()
    rows = np.array(list(range(0, cu[4], 5)) + list(range(cu[4], cu[-1])), dtype=np.int32)
    outs, kc, vc = run_gpu(w, fused_prefill=True)
    assert_status_ok()
    ref, kr, vr = run_oracle(w, rows_for=lambda i: rows)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    mask = np.zeros(cu[-1], bool)
    mask[rows] = True
    assert_attn_close(outs[0], ref[0], w.name, mask=mask)


@pytest.mark.parametrize("hq,hkv,d,bs", [(4, 2, 64, 16), (16, 8, 128, 256), (32, 4, 64, 32)])
def test_append_mixed_chunks_and_decode_rows(hq, hkv, d, bs):
    chunks = [(40, 0), (300, 133), (97, 96), (513, 256), (129, 1)]
    dec = [1, 2, 17, 200, 1000, 64, 65]
    nb = sum(W.num_blocks_for(L, bs) for L, _ in chunks) + sum(W.num_blocks_for(L, bs) for L in dec) + 5
    _check(W.mixed_workload(f"mixed_append_{hq}_{hkv}_{d}_{bs}", chunks, dec, hq, hkv, d, bs, nb))


def test_append_graph_replay_and_repeated_calls():
    """The cooperative launch captured in a CUDA graph and replayed (the
    store counter must start from zero on every replay), and 70 eager calls in
    a row (every counter slot used more than once)."""
    w = W.config3_prefill()
    st, a = w.steps[0].store, w.steps[0].attn
    m = a.meta
    kc, vc = gpu_pool(w)
    for s in w.setup:
        kvp.kv_store(s.k.cuda(), s.v.cuda(), s.slot_mapping.cuda(), kc, vc)
    args = [t.cuda() for t in (a.q, st.k, st.v, st.slot_mapping, m.cu_seqlens_q, m.cu_seqlens_k)]
    bt = m.block_tables.cuda()
    out = torch.empty((args[0].shape[0], w.num_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")

    def call():
        kvp.attn_prefill_varlen_append(args[0], args[1], args[2], args[3], args[4], args[5], m.max_seqlen_q,
                                       m.max_seqlen_k, kc, vc, block_tables=bt, softmax_scale=w.scale, out=out)

    call()
    torch.cuda.synchronize()
    first = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    for _ in range(70):
        call()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    assert_status_ok()
    ref, kr, vr = run_oracle(w)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    assert_attn_close(first, ref[0], "graph replay")


def test_append_flags_bad_slots_and_packed_prefix():
    """A slot past the pool stores nothing and records KVP_ERR_DEVICE_DATA;
    packed mode (no block tables) with a cached prefix (k_len != q_len) is
    reported the same way."""
    w = W.prefill_workload("pfa_bad", [300, 200], [0, 0], 4, 2, 64, 16, 40)
    st, a = w.steps[0].store, w.steps[0].attn
    m = a.meta
    kc, vc = gpu_pool(w)
    slots = st.slot_mapping.clone()
    slots[5] = 40 * 16 + 3
    kvp.attn_prefill_varlen_append(a.q.cuda(), st.k.cuda(), st.v.cuda(), slots.cuda(), m.cu_seqlens_q.cuda(),
                                   m.cu_seqlens_k.cuda(), m.max_seqlen_q, m.max_seqlen_k, kc, vc)
    assert kvp.device_status() == -6
    kr, vr = oracle_pool(w)
    good = slots.clone()
    good[5] = -1
    oracle.kv_store(st.k, st.v, good, kr, vr)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    cu_k = m.cu_seqlens_k.clone()
    cu_k[1:] += 16  # a "cached prefix" of 16 keys per sequence without block tables
    kvp.attn_prefill_varlen_append(a.q.cuda(), st.k.cuda(), st.v.cuda(), st.slot_mapping.cuda(),
                                   m.cu_seqlens_q.cuda(), cu_k.cuda(), m.max_seqlen_q, m.max_seqlen_k + 16,
                                   kc, vc)
    assert kvp.device_status() == -6
