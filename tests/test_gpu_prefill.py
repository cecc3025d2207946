"""GPU parity: attn_prefill_varlen (tcgen05 path) against the CPU oracle, and the
whole store -> prefill -> decode pipeline of the tiny configuration."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

from parity import assert_attn_close, assert_status_ok, run_gpu, run_oracle, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    kvp.device_status()
    yield
    assert_status_ok()


def _check(w, rows_for=None):
    outs, kc, vc = run_gpu(w)
    ref, kr, vr = run_oracle(w, rows_for=rows_for)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr), "cache differs after kv_store"
    res = []
    for i, (o, r) in enumerate(zip(outs, ref)):
        mask = None if rows_for is None or not w.steps[i].is_prefill else rows_for(i)
        res.append(assert_attn_close(o, r, f"{w.name} step {i}", mask))
    return res


def test_config1_tiny_pipeline():
    """Store the cached prefix, prefill 17 + 284 tokens (paged: the second prompt
    has a cached block), then 4 decode steps; bs 16, d 64, Hq 2 / Hkv 1."""
    _check(W.config1_tiny())


def test_config3_full_size():
    """8 prompts U[256, 2048], 0-2 cached blocks each, Qwen3-8B heads, bs 256."""
    _check(W.config3_prefill())


@pytest.mark.parametrize("hq,hkv,d,bs,lens,cached", [
    (2, 2, 64, 16, [1, 2, 129, 300], [0, 0, 0, 0]),            # G=1, packed (no prefix)
    (4, 2, 128, 16, [45, 200, 333], [1, 0, 4]),                  # G=2, paged, bs 16
    (8, 2, 128, 32, [640, 70], [5, 2]),                          # G=4, bs 32
    (16, 2, 64, 256, [1000, 257, 256], [1, 0, 0]),               # G=8, d 64
    (32, 8, 128, 256, [2048, 1, 130], [7, 0, 0]),                # Qwen3-8B heads, long prefix
    (16, 8, 128, 128, [777, 128, 129], [2, 0, 1]),               # bs 128
    (8, 8, 128, 64, [300, 301, 302, 303, 304], [0, 1, 2, 3, 4]),
    (4, 1, 64, 16, [17, 300], [0, 1]),
    (16, 8, 128, 256, [100, 900, 2000, 37], [0, 0, 0, 0]),       # packed, several kv tiles
])
def test_prefill_shapes(hq, hkv, d, bs, lens, cached):
    nb = sum(W.num_blocks_for(L, bs) for L in lens) + 5
    w = W.prefill_workload(f"pf_{hq}_{hkv}_{d}_{bs}", lens, cached, hq, hkv, d, bs, nb)
    _check(w)


def _schedule_case(kind):
    rng = np.random.default_rng({"cu_global": 1, "cu_global_rr": 2, "at_limit": 3, "over_limit": 4}[kind])
    if kind == "cu_global":  # 530 short prompts: cu_seqlens stay in global memory, cost order kept
        hq, hkv, d, bs = 4, 2, 128, 16
        lens = rng.integers(1, 101, size=530).tolist()
    elif kind == "cu_global_rr":  # 600 prompts, one long: global cu_seqlens and round-robin order
        hq, hkv, d, bs = 8, 2, 64, 32
        lens = rng.integers(1, 41, size=599).tolist() + [1500]
    else:  # 64 (at the limit) or 65 (past it) prompts, one of 4096 tokens: 64 pair ranks each
        hq, hkv, d, bs = 4, 1, 64, 64
        n = 64 if kind == "at_limit" else 65
        lens = [4096] + rng.integers(1, 201, size=n - 1).tolist()
    cached = [int(rng.integers(0, (L - 1) // bs + 1)) if L > bs and rng.random() < 0.5 else 0
              for L in lens]
    nb = sum(W.num_blocks_for(L, bs) for L in lens) + 3
    return W.prefill_workload(f"sched_{kind}", lens, cached, hq, hkv, d, bs, nb)


@pytest.mark.parametrize("kind,dynamic,cu_in_smem", [("cu_global", True, False),
                                                     ("cu_global_rr", False, False),
                                                     ("at_limit", True, True),
                                                     ("over_limit", False, True)])
def test_prefill_schedule_capacity_fallbacks(kind, dynamic, cu_in_smem):
    """The per-CTA schedule holds cu_seqlens for at most 519 sequences and
    the cost order for at most 4096 (pair rank, sequence) entries; past them
    the kernel reads cu_seqlens from global memory and takes items
    round-robin.  Each side of both limits against the oracle."""
    w = _schedule_case(kind)
    m = w.steps[0].attn.meta
    g = w.num_heads // w.num_kv_heads
    num_seqs = m.cu_seqlens_q.numel() - 1
    max_pairs = -(-m.max_seqlen_q // (2 * (128 // g)))
    assert (max_pairs * num_seqs <= 4096) == dynamic
    assert (num_seqs + 1 <= 520) == cu_in_smem
    _check(w)


def test_prefill_fully_cached_prompt_has_no_rows():
    """A block-aligned prompt whose every block hit the prefix cache has
    q_len 0; the other sequences are unaffected."""
    w = W.prefill_workload("fully_cached", [64, 100], [4, 1], 4, 2, 64, 16, 32)
    m = w.steps[0].attn.meta
    assert m.cu_seqlens_q.tolist()[:2] == [0, 0]
    _check(w)


def test_prefill_then_decode_matches_oracle_qwen3_shapes():
    w = W.prefill_workload("pf_then_decode", [300, 513, 1200], [1, 2, 0], 16, 8, 128, 256, 32,
                           extra_decode_steps=3)
    _check(w)


def test_prefill_out_of_range_block_is_flagged():
    w = W.prefill_workload("bad", [100, 60], [1, 1], 4, 2, 128, 16, 32)
    kc, vc = w.new_cache("cuda")
    for st in w.setup + [w.steps[0].store]:
        kvp.kv_store(st.k.cuda(), st.v.cuda(), st.slot_mapping.cuda(), kc, vc)
    a = w.steps[0].attn
    bt = a.meta.block_tables.clone()
    bt[0, 2] = 9999
    kvp.attn_prefill_varlen(a.q.cuda(), a.meta.cu_seqlens_q.cuda(), a.meta.cu_seqlens_k.cuda(),
                            a.meta.max_seqlen_q, a.meta.max_seqlen_k, k_cache=kc, v_cache=vc,
                            block_tables=bt.cuda())
    assert kvp.device_status() == -6


@pytest.mark.parametrize("cached_blocks,hq,hkv", [(0, 16, 8), (2, 16, 8), (2, 32, 8), (1, 8, 1)])
def test_prefill_scores_growing_across_tiles(cached_blocks, hq, hkv):
    """Keys whose scores rise by ~10 (log2 units) per 128-key tile: the running
    max grows past the lazy-rescale threshold on every tile, so the O / row-sum
    rescale path runs (warp-wide) on every tile of every row."""
    L, d, bs = 900, 128, 128
    nb = W.num_blocks_for(L, bs) + 3
    w = W.prefill_workload(f"rescale_{cached_blocks}_{hq}_{hkv}", [L], [cached_blocks], hq, hkv, d,
                           bs, nb)
    g = torch.Generator().manual_seed(31)
    c = cached_blocks * bs

    def keys(pos):
        p = torch.tensor(pos, dtype=torch.float32)[:, None, None]
        return (0.02 * p * torch.ones((len(pos), hkv, d)) +
                0.1 * torch.randn((len(pos), hkv, d), generator=g)).to(torch.bfloat16)

    if c:
        w.setup[0].k.copy_(keys(list(range(c))))
    st, a = w.steps[0].store, w.steps[0].attn
    st.k.copy_(keys(list(range(c, L))))
    a.q.copy_((0.25 + 0.05 * torch.randn(a.q.shape, generator=g)).to(torch.bfloat16))
    _check(w)


def _prefill_inputs(w):
    import types
    from parity import gpu_pool
    kc, vc = gpu_pool(w)
    for st in w.setup:
        kvp.kv_store(st.k.cuda(), st.v.cuda(), st.slot_mapping.cuda(), kc, vc)
    s, a = w.steps[0].store, w.steps[0].attn
    kvp.kv_store(s.k.cuda(), s.v.cuda(), s.slot_mapping.cuda(), kc, vc)
    m = a.meta
    return types.SimpleNamespace(
        q=a.q.cuda(), k=a.k.cuda(), v=a.v.cuda(), kc=kc, vc=vc, cq=m.cu_seqlens_q.cuda(),
        ck=m.cu_seqlens_k.cuda(), mq=m.max_seqlen_q, mk=m.max_seqlen_k,
        bt=None if m.block_tables is None else m.block_tables.cuda(),
        out=torch.empty_like(a.q.cuda()))


def _prefill_call(x, w):
    kvp.attn_prefill_varlen(x.q, x.cq, x.ck, x.mq, x.mk, k=x.k, v=x.v, k_cache=x.kc, v_cache=x.vc,
                            block_tables=x.bt, num_kv_heads=w.num_kv_heads, softmax_scale=w.scale,
                            out=x.out)


def test_prefill_graph_replays_repeat_the_schedule():
    """The work counter of a launch is reset by its last CTA, so a captured
    prefill call gives the full result on every replay."""
    w = W.prefill_workload("graph_replay", [700, 1500, 90, 2048], [1, 0, 0, 2], 32, 8, 128, 256, 64)
    x = _prefill_inputs(w)
    ref, _, _ = run_oracle(w)
    _prefill_call(x, w)  # first use outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        _prefill_call(x, w)
    for rep in range(3):
        x.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_status_ok()
        assert_attn_close(x.out, ref[0], f"graph replay {rep}")


def test_prefill_many_launches_reuse_counter_slots():
    """More launches than counter slots: every slot is used again with a new
    epoch; the last launch still covers every item."""
    w = W.prefill_workload("many_launches", [300, 33, 1100], [0, 0, 1], 16, 8, 128, 256, 16)
    x = _prefill_inputs(w)
    ref, _, _ = run_oracle(w)
    for i in range(140):
        if i == 139:
            x.out.fill_(float("nan"))
        _prefill_call(x, w)
    torch.cuda.synchronize()
    assert_status_ok()
    assert_attn_close(x.out, ref[0], "launch 140")


def test_prefill_concurrent_streams_use_separate_counters():
    """Two prefill calls in flight at once on two streams take different
    counter slots; both results are complete."""
    w1 = W.prefill_workload("streams_a", [900, 400, 1500], [1, 0, 2], 32, 8, 128, 256, 32)
    w2 = W.prefill_workload("streams_b", [2048, 77], [0, 0], 16, 8, 128, 256, 16)
    x1, x2 = _prefill_inputs(w1), _prefill_inputs(w2)
    r1, _, _ = run_oracle(w1)
    r2, _, _ = run_oracle(w2)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(20):
        with torch.cuda.stream(s1):
            _prefill_call(x1, w1)
        with torch.cuda.stream(s2):
            _prefill_call(x2, w2)
    torch.cuda.synchronize()
    assert_status_ok()
    assert_attn_close(x1.out, r1[0], "stream 1")
    assert_attn_close(x2.out, r2[0], "stream 2")
