"""GPU checks of the merge of cut sequences: a sequence that crosses CTA
ranges of the decode's flat split leaves partials that the merge kernel
combines.  Many calls in a row, two calls in flight on two streams (each
with its own workspace), and a captured call replayed, where one sequence
crosses every CTA range; each output equal bit for bit to the first call's
and checked against the oracle."""
import pytest
import torch

import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

from parity import assert_attn_close, assert_status_ok, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    kvp.device_status()
    yield
    assert_status_ok()


def _inputs(w):
    """The workload's cache after its setup and store, and its decode inputs on the device."""
    outs, kc, vc = run_gpu(w)
    a = w.steps[0].attn
    m = a.meta
    x = dict(q=a.q.cuda(), kc=kc, vc=vc, bt=m.block_tables.cuda(), ctx=m.context_lens.cuda(),
             max_ctx=m.max_context_len)
    ws = torch.empty(kvp.attn_decode_workspace_size(m.context_lens.numel(), w.num_heads, w.head_dim,
                                                    m.max_context_len, w.block_size),
                     dtype=torch.uint8, device="cuda")
    return x, ws, outs[0]


def _call(x, w, ws, out):
    kvp.attn_decode_paged(x["q"], x["kc"], x["vc"], x["bt"], x["ctx"], x["max_ctx"],
                          softmax_scale=w.scale, workspace=ws, out=out)


def test_decode_many_calls_in_a_row():
    """150 calls in a row: the last output equals the first bit for bit and
    the oracle."""
    w = W.decode_workload("merge_rows", [700, 2500, 90, 4000, 1300, 3333, 17, 2048], 16, 8, 128, 256, 64)
    x, ws, first = _inputs(w)
    out = torch.empty_like(first)
    for i in range(150):
        if i == 149:
            out.fill_(float("nan"))
        _call(x, w, ws, out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    ref, _, _ = run_oracle(w)
    assert_attn_close(out, ref[0], "call 150")


def test_decode_two_calls_in_flight_on_two_streams():
    w1 = W.decode_workload("merge_s1", [3000, 1500, 4096, 700], 32, 8, 128, 256, 64)
    w2 = W.decode_workload("merge_s2", [5000, 333, 2222], 16, 8, 128, 256, 64)
    x1, ws1, f1 = _inputs(w1)
    x2, ws2, f2 = _inputs(w2)
    o1, o2 = torch.empty_like(f1), torch.empty_like(f2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(20):
        with torch.cuda.stream(s1):
            _call(x1, w1, ws1, o1)
        with torch.cuda.stream(s2):
            _call(x2, w2, ws2, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), f1.view(torch.int16))
    assert torch.equal(o2.view(torch.int16), f2.view(torch.int16))
    r1, _, _ = run_oracle(w1)
    r2, _, _ = run_oracle(w2)
    assert_attn_close(o1, r1[0], "stream 1")
    assert_attn_close(o2, r2[0], "stream 2")


def test_decode_graph_replays_merge_every_time():
    """One sequence crosses every CTA range; every replay of the captured call
    merges all its parts again."""
    w = W.decode_workload("merge_graph", [65536, 100, 9000], 16, 8, 128, 256, 300)
    x, ws, first = _inputs(w)
    out = torch.empty_like(first)
    _call(x, w, ws, out)  # first use outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _call(x, w, ws, out)
    torch.cuda.current_stream().wait_stream(s)
    ref, _, _ = run_oracle(w)
    for rep in range(5):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), first.view(torch.int16)), f"replay {rep}"
    assert_attn_close(out, ref[0], "graph replay")
