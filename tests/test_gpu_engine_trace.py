"""GPU replay of the engine-step trace (config: 256 requests, prompts and
outputs U[100, 1024], 28 layers of Qwen3-0.6B attention shape, bs 256,
768-block pool, max_num_batched_tokens 16384, max_num_seqs 512): every step
calls kv_store and prefill or decode attention on all 28 layers, with per-layer
Q/K/V drawn from a generator keyed on (step, layer).  The oracle follows layers
0 and 27: it replays every store (the caches must match bit for bit at the
end) and checks attention on a seeded sample of steps (all sequences of a
decode step; a row sample of a prefill step)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import engine_trace as E

from parity import BF16_NAN, assert_attn_close, u16

pytestmark = pytest.mark.gpu

LAYERS, HQ, HKV, D, BS, NB = 28, 16, 8, 128, 256, 768
CHECK_LAYERS = (0, 27)


def layer_inputs(step, layer, n, device):
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * step + 7919 * layer + 17)
    q = torch.randn((n, HQ, D), generator=g, device=device).to(torch.bfloat16)
    k = torch.randn((n, HKV, D), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((n, HKV, D), generator=g, device=device).to(torch.bfloat16)
    return q, k, v


def test_config5_trace_replay_all_layers():
    dev = torch.device("cuda")
    kv_cache = torch.full((2, LAYERS, NB, BS, HKV, D), float("nan"), dtype=torch.bfloat16, device=dev)
    ora = {l: (np.full((NB, BS, HKV, D), BF16_NAN, np.uint16), np.full((NB, BS, HKV, D), BF16_NAN, np.uint16))
           for l in CHECK_LAYERS}
    scale = D ** -0.5
    rng = np.random.default_rng(5)
    checked_decode = checked_prefill = 0
    n_steps = 0
    for st, sched in E.engine_trace():
        m = st.meta
        n = st.num_new_tokens
        slots = m.slot_mapping.to(dev)
        check = st.index in (0, 1) or rng.random() < 0.006
        for layer in range(LAYERS):
            kc, vc = kv_cache[0, layer], kv_cache[1, layer]
            q, k, v = layer_inputs(st.index, layer, n, dev)
            kvp.kv_store(k, v, slots, kc, vc)
            if st.is_prefill:
                bt = None if m.block_tables is None else m.block_tables.to(dev)
                out = kvp.attn_prefill_varlen(q, m.cu_seqlens_q.to(dev), m.cu_seqlens_k.to(dev),
                                              m.max_seqlen_q, m.max_seqlen_k, k=k, v=v, k_cache=kc,
                                              v_cache=vc, block_tables=bt, num_kv_heads=HKV,
                                              softmax_scale=scale)
            else:
                out = kvp.attn_decode_paged(q, kc, vc, m.block_tables.to(dev), m.context_lens.to(dev),
                                            m.max_context_len, softmax_scale=scale)
            if layer in CHECK_LAYERS:
                okc, ovc = ora[layer]
                oracle.kv_store(k.cpu(), v.cpu(), m.slot_mapping, okc, ovc)
                if check:
                    if st.is_prefill:
                        rows = np.sort(rng.choice(n, size=min(n, 192), replace=False))
                        if m.block_tables is None:
                            ref = oracle.prefill(q.cpu(), m.cu_seqlens_q, m.cu_seqlens_k, HQ, HKV, scale,
                                                 k=k.cpu(), v=v.cpu(), rows=rows)
                        else:
                            ref = oracle.prefill(q.cpu(), m.cu_seqlens_q, m.cu_seqlens_k, HQ, HKV, scale,
                                                 k_cache=okc, v_cache=ovc, block_tables=m.block_tables,
                                                 rows=rows)
                        assert_attn_close(out, ref, f"step {st.index} layer {layer} (prefill)", rows)
                        checked_prefill += 1
                    else:
                        ref = oracle.decode(q.cpu(), okc, ovc, m.block_tables, m.context_lens, HQ, HKV,
                                            scale)
                        assert_attn_close(out, ref, f"step {st.index} layer {layer} (decode)")
                        checked_decode += 1
        n_steps += 1
    torch.cuda.synchronize()
    assert kvp.device_status() == 0
    assert n_steps > 1000 and sched.preemptions > 0
    assert checked_prefill >= 2 and checked_decode >= 2
    for layer in CHECK_LAYERS:
        okc, ovc = ora[layer]
        assert np.array_equal(u16(kv_cache[0, layer]), okc), f"layer {layer} K cache"
        assert np.array_equal(u16(kv_cache[1, layer]), ovc), f"layer {layer} V cache"
