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
        # The same step with its metadata packed for the bucket in pinned
        # memory, one copy (q/k/v already in the graph's buffers): the same
        # bits, and the cache rows stored again unchanged.
        first = out.clone()
        packed = graphs.pack(b, st.slot_mapping, m.block_tables, m.context_lens,
                             out=torch.empty((graphs.meta.numel(),), dtype=torch.int32,
                                             pin_memory=True))
        graphs.out.fill_(float("nan"))
        out2 = graphs.run_packed(b, packed)
        torch.cuda.synchronize()
        assert_status_ok()
        assert torch.equal(out2.view(torch.int16), first.view(torch.int16)), b
        assert torch.all(graphs.out[b:pb].float() == 0)
        assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr), b


def test_layered_graph_decode_matches_oracle():
    """Three layers in one graph per bucket (the engine's whole-model decode
    capture): each layer's cache after the replay is bit-exact and its output
    matches the oracle's store-then-decode on that layer."""
    import oracle
    from paged_kv_cache_125_gb300.graphs import LayeredDecodeGraphs
    from parity import oracle_pool

    hq, hkv, d, bs, layers = 8, 4, 128, 16, 3
    max_bs, max_blocks = 32, 10
    nb = max_bs * max_blocks + 4
    caches = [(torch.empty((nb, bs, hkv, d), dtype=torch.bfloat16, device="cuda"),
               torch.empty((nb, bs, hkv, d), dtype=torch.bfloat16, device="cuda")) for _ in range(layers)]
    graphs = LayeredDecodeGraphs(caches, hq, max_blocks, max_bs=max_bs)
    rng = np.random.default_rng(11)
    for b in (1, 6, 32, 3):
        ctx = rng.integers(1, max_blocks * bs + 1, size=b).tolist()
        w = W.decode_workload(f"layered_b{b}", ctx, hq, hkv, d, bs, nb)
        st, a = w.steps[0].store, w.steps[0].attn
        qs = [(a.q.float() * (1 + 0.5 * layer)).to(torch.bfloat16) for layer in range(layers)]
        for layer, (kc, vc) in enumerate(caches):
            kc.fill_(float("nan"))
            vc.fill_(float("nan"))
            w.place_history(kc, vc)
            graphs.q[layer, :b].copy_(qs[layer])
            graphs.k[layer, :b].copy_(st.k)
            graphs.v[layer, :b].copy_(st.v)
        pb = graphs.run(b, st.slot_mapping.cuda(), a.meta.block_tables.cuda(), a.meta.context_lens.cuda())
        torch.cuda.synchronize()
        assert_status_ok()
        assert pb == graphs.bucket(b)
        kr, vr = oracle_pool(w)
        oracle.kv_store(st.k, st.v, st.slot_mapping, kr, vr)
        for layer, (kc, vc) in enumerate(caches):
            assert np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr), (b, layer)
            ref = oracle.decode(qs[layer], kr, vr, a.meta.block_tables, a.meta.context_lens, hq, hkv,
                                w.scale)
            assert_attn_close(graphs.out[layer, :b], ref, f"layered decode b={b} layer {layer}")
        # the packed-metadata path replays the same bucket and gives the same bits
        first = graphs.out[:, :b].clone()
        graphs.out.fill_(float("nan"))
        packed = graphs.pack(b, st.slot_mapping, a.meta.block_tables, a.meta.context_lens)
        assert graphs.run_packed(b, packed.pin_memory()) == pb
        torch.cuda.synchronize()
        assert_status_ok()
        assert torch.equal(graphs.out[:, :b].view(torch.int16), first.view(torch.int16)), b
