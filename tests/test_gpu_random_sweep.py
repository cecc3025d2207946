"""Seeded random sweep of shapes against the oracle (property-style): random
head counts, head_dim, block size, sequence count, lengths (including 1 and
block-aligned ones) and cached prefixes, for prefill followed by decode."""
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
