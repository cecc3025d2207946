"""Seeded random sweep of shapes against the oracle (property-style): random
head counts, head_dim, block size, sequence count, lengths (including 1 and
block-aligned ones) and cached prefixes, for prefill followed by decode,
with the stores as separate calls and fused into the attention calls; and
random mixed steps (chunks and decode rows through attn_mixed_step)."""
import numpy as np
import pytest

import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

from parity import assert_attn_close, assert_status_ok, run_gpu, run_oracle, u16

pytestmark = pytest.mark.gpu


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32, 64, 128, 256]))
    nseq = int(rng.integers(1, 7))
    lens, cached = [], []
    for _ in range(nseq):
        kind = rng.random()
        if kind < 0.15:
            L = 1
        elif kind < 0.3:
            L = bs * int(rng.integers(1, 5))
        else:
            L = int(rng.integers(2, 1500))
        lens.append(L)
        cached.append(int(rng.integers(0, (L - 1) // bs + 1)) if L > 1 and rng.random() < 0.6 else 0)
    steps = int(rng.integers(0, 3))
    nb = sum(W.num_blocks_for(L + steps, bs) for L in lens) + int(rng.integers(0, 9))
    return W.prefill_workload(f"sweep{seed}", lens, cached, g * hkv, hkv, d, bs, nb,
                              extra_decode_steps=steps)


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes(seed):
    w = _random_case(seed)
    kvp.device_status()
    outs, kc, vc = run_gpu(w)
    ref, kr, vr = run_oracle(w)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    for i, (o, r) in enumerate(zip(outs, ref)):
        assert_attn_close(o, r, f"{w.name} step {i}")
    assert_status_ok()


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes_fused_stores(seed):
    """The same seeded cases with every step's store fused into its attention
    call (attn_prefill_varlen_append, attn_decode_paged_append)."""
    w = _random_case(seed)
    kvp.device_status()
    outs, kc, vc = run_gpu(w, fused_decode=True, fused_prefill=True)
    ref, kr, vr = run_oracle(w)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    for i, (o, r) in enumerate(zip(outs, ref)):
        assert_attn_close(o, r, f"{w.name} (fused) step {i}")
    assert_status_ok()


def _random_mixed_case(seed):
    rng = np.random.default_rng(5000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32, 64, 128, 256]))
    chunks = []
    for _ in range(int(rng.integers(1, 5))):
        total = int(rng.integers(2, 2500))
        cached = int(rng.integers(0, total)) if rng.random() < 0.7 else 0
        chunks.append((total, cached))
    dec = [int(x) for x in rng.integers(1, 3000, int(rng.integers(1, 40)))]
    nb = sum(W.num_blocks_for(L, bs) for L, _ in chunks) + sum(W.num_blocks_for(L, bs) for L in dec) + 3
    sms = int(rng.choice([0, 0, 8, 40, 100, 150]))
    return W.mixed_workload(f"msweep{seed}", chunks, dec, g * hkv, hkv, d, bs, nb), len(dec), sms


@pytest.mark.parametrize("seed", range(12))
def test_random_mixed_steps(seed):
    """attn_mixed_step on seeded random chunks (cached prefixes ending
    anywhere, inside a block or not) and decode rows, with a random share of
    the SMs for the decode rows: caches bit-exact, every row against the
    oracle."""
    import torch
    from parity import gpu_pool
    w, nd, sms = _random_mixed_case(seed)
    kvp.device_status()
    kc, vc = gpu_pool(w)
    st, a = w.steps[0].store, w.steps[0].attn
    m = a.meta
    out = kvp.attn_mixed_step(a.q.cuda(), st.k.cuda(), st.v.cuda(), st.slot_mapping.cuda(),
                              m.cu_seqlens_q.cuda(), m.cu_seqlens_k.cuda(), m.max_seqlen_q, m.max_seqlen_k,
                              kc, vc, m.block_tables.cuda(), nd, decode_sms=sms, softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert_status_ok()
    ref, kr, vr = run_oracle(w)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    assert_attn_close(out, ref[0], w.name)
