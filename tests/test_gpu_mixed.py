"""Chunked prefill mixed with decode rows in one varlen paged prefill call
(every decode row is a sequence with q_len 1; chunk boundaries may fall inside
a block), against the oracle through the C ABI."""
import numpy as np
import pytest
import torch

from paged_kv_cache_125_gb300 import workloads as W

from parity import assert_attn_close, assert_status_ok, run_gpu, run_oracle, u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hkv,d,bs", [(4, 2, 64, 16), (16, 8, 128, 256), (8, 1, 128, 64),
                                         (32, 4, 64, 32)])
def test_mixed_chunks_and_decode_rows(hq, hkv, d, bs):
    chunks = [(40, 0), (300, 133), (97, 96), (513, 256), (129, 1)]
    dec = [1, 2, 17, 200, 1000, 64, 65]
    nb = sum(W.num_blocks_for(L, bs) for L, _ in chunks) + sum(W.num_blocks_for(L, bs) for L in dec) + 5
    w = W.mixed_workload(f"mixed_{hq}_{hkv}_{d}_{bs}", chunks, dec, hq, hkv, d, bs, nb)
    outs, kc, vc = run_gpu(w)
    ref, kr, vr = run_oracle(w)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    assert_attn_close(outs[0], ref[0], w.name)
    assert_status_ok()


def test_mixed_step_full_size_sampled():
    """The bench's mixed step (4 prefill chunks of a 32/8/128 model + 128
    decode rows): every decode row and every 5th chunk row against the
    oracle; caches bit-exact."""
    w = W.mixed_step_workload()
    m = w.steps[0].attn.meta
    cu = m.cu_seqlens_q.tolist()
    n_chunk_rows = cu[4]
    rows = np.array(list(range(0, n_chunk_rows, 5)) + list(range(n_chunk_rows, cu[-1])), dtype=np.int32)
    outs, kc, vc = run_gpu(w)
    ref, kr, vr = run_oracle(w, rows_for=lambda i: rows)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    mask = np.zeros(cu[-1], bool)
    mask[rows] = True
    assert_attn_close(outs[0], ref[0], w.name, mask=mask)
    assert_status_ok()
