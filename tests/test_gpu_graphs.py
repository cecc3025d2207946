"""Graph-replayed decode with batch-size buckets (the engine's CUDA-graph
path, "nano-vLLM-1" ModelRunner): one capture per bucket, steps of several
sizes padded to their bucket (slot -1, context 0), against the oracle."""
import numpy as np
import pytest
import torch

from paged_kv_cache_125_gb300 import workloads as W
from paged_kv_cache_125_gb300.graphs import DecodeGraphs

from parity import assert_attn_close, assert_status_ok, run_oracle, u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hkv,d,bs", [(16, 8, 128, 256), (4, 2, 64, 16)])
def test_bucketed_graph_decode_matches_oracle(hq, hkv, d, bs):
    max_bs, max_blocks = 64, 12
    nb = max_bs * max_blocks + 8
    kc = torch.empty((nb, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    graphs = DecodeGraphs(kc, vc, hq, max_blocks, max_bs=max_bs)
    assert graphs.buckets == [1, 2, 4, 8, 16, 32, 48, 64]
    rng = np.random.default_rng(bs)
    for b in (1, 3, 8, 17, 64, 5):
        ctx = rng.integers(1, max_blocks * bs + 1, size=b).tolist()
        w = W.decode_workload(f"graph_b{b}", ctx, hq, hkv, d, bs, nb)
        kc.fill_(float("nan"))
        vc.fill_(float("nan"))
        w.place_history(kc, vc)
        st, m = w.steps[0].store, w.steps[0].attn.meta
        out = graphs.run(w.steps[0].attn.q.cuda(), st.k.cuda(), st.v.cuda(), st.slot_mapping.cuda(),
                         m.block_tables.cuda(), m.context_lens.cuda())
        torch.cuda.synchronize()
        assert_status_ok()
        ref, kr, vr = run_oracle(w)
        assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr), b
        assert_attn_close(out, ref[0], f"bucketed decode b={b} (bucket {graphs.bucket(b)})")
        # padding rows of the bucket produced zeros and wrote nothing
        pb = graphs.bucket(b)
        assert torch.all(graphs.out[b:pb].float() == 0)
