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


# --------------------------------------------------------------------------- attn_mixed_step

def _mixed_call(w, num_decode, decode_sms=0, kc=None, vc=None):
    import paged_kv_cache_125_gb300 as kvp
    from parity import gpu_pool
    if kc is None:
        kc, vc = gpu_pool(w)
    st, a = w.steps[0].store, w.steps[0].attn
    m = a.meta
    out = kvp.attn_mixed_step(a.q.cuda(), st.k.cuda(), st.v.cuda(), st.slot_mapping.cuda(),
                              m.cu_seqlens_q.cuda(), m.cu_seqlens_k.cuda(), m.max_seqlen_q, m.max_seqlen_k,
                              kc, vc, m.block_tables.cuda(), num_decode, decode_sms=decode_sms,
                              softmax_scale=w.scale)
    torch.cuda.synchronize()
    return out, kc, vc


@pytest.mark.parametrize("hq,hkv,d,bs,decode_sms", [(4, 2, 64, 16, 0), (16, 8, 128, 256, 0),
                                                    (8, 1, 128, 64, 40), (32, 4, 64, 32, 120),
                                                    (32, 8, 128, 256, 16)])
def test_mixed_step_chunks_beside_decode_rows(hq, hkv, d, bs, decode_sms):
    """attn_mixed_step: the chunks through the fused store + prefill, the
    decode rows (the last sequences, q_len 1) through the decode kernel with
    the store fused, side by side; caches bit-exact, outputs against the
    oracle's store-then-prefill."""
    chunks = [(40, 0), (300, 133), (97, 96), (513, 256), (129, 1)]
    dec = [1, 2, 17, 200, 1000, 64, 65]
    nb = sum(W.num_blocks_for(L, bs) for L, _ in chunks) + sum(W.num_blocks_for(L, bs) for L in dec) + 5
    w = W.mixed_workload(f"mixed_step_{hq}_{hkv}_{d}_{bs}", chunks, dec, hq, hkv, d, bs, nb)
    out, kc, vc = _mixed_call(w, len(dec), decode_sms)
    assert_status_ok()
    ref, kr, vr = run_oracle(w)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    assert_attn_close(out, ref[0], w.name)


@pytest.mark.parametrize("which", ["decode_only", "chunks_only"])
def test_mixed_step_one_kind_of_rows(which):
    chunks = [] if which == "decode_only" else [(40, 0), (300, 133), (513, 256)]
    dec = [3, 17, 200, 1000] if which == "decode_only" else []
    nb = sum(W.num_blocks_for(L, 16) for L, _ in chunks) + sum(W.num_blocks_for(L, 16) for L in dec) + 5
    w = W.mixed_workload(f"mixed_{which}", chunks, dec, 16, 8, 128, 16, nb)
    out, kc, vc = _mixed_call(w, len(dec))
    assert_status_ok()
    ref, kr, vr = run_oracle(w)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    assert_attn_close(out, ref[0], w.name)


def test_mixed_step_full_size_sampled_and_graph_replay():
    """The bench's mixed step (4 chunks of a 32/8/128 model + 128 decode rows)
    through attn_mixed_step, eager and as a CUDA-graph replay (the chain of
    programmatic dependent launches captured as one graph): every decode row
    and every 5th chunk row against the oracle, caches bit-exact, the replay
    bit-identical to the eager call."""
    import paged_kv_cache_125_gb300 as kvp
    from parity import gpu_pool
    w = W.mixed_step_workload()
    st, a = w.steps[0].store, w.steps[0].attn
    m = a.meta
    cu = m.cu_seqlens_q.tolist()
    rows = np.array(list(range(0, cu[4], 5)) + list(range(cu[4], cu[-1])), dtype=np.int32)
    out, kc, vc = _mixed_call(w, 128)
    assert_status_ok()
    ref, kr, vr = run_oracle(w, rows_for=lambda i: rows)
    assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)
    mask = np.zeros(cu[-1], bool)
    mask[rows] = True
    assert_attn_close(out, ref[0], w.name, mask=mask)
    args = [t.cuda() for t in (a.q, st.k, st.v, st.slot_mapping, m.cu_seqlens_q, m.cu_seqlens_k,
                               m.block_tables)]
    ws = torch.empty(kvp.attn_decode_workspace_size(128, 32, 128, m.max_seqlen_k, 256), dtype=torch.uint8,
                     device="cuda")
    o2 = torch.empty_like(out)

    def call():
        kvp.attn_mixed_step(args[0], args[1], args[2], args[3], args[4], args[5], m.max_seqlen_q, m.max_seqlen_k,
                            kc, vc, args[6], 128, softmax_scale=w.scale, workspace=ws, out=o2)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        o2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o2.view(torch.int16), out.view(torch.int16))
    assert_status_ok()


def test_mixed_step_flags_a_decode_row_with_two_query_rows():
    """A trailing 'decode row' that queries two tokens is reported
    (KVP_ERR_DEVICE_DATA); a valid split of the same shapes is not."""
    import paged_kv_cache_125_gb300 as kvp
    good = W.mixed_workload("mixed_good", [(40, 0), (200, 199)], [300], 4, 2, 64, 16, 64)
    _mixed_call(good, 1)
    assert kvp.device_status() == 0
    bad = W.mixed_workload("mixed_bad", [(40, 0), (300, 298)], [], 4, 2, 64, 16, 64)
    _mixed_call(bad, 1)
    assert kvp.device_status() == -6
