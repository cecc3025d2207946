"""GPU replay of the engine-step trace (256 requests, prompts and outputs
U[100, 1024], 28 layers of Qwen3-0.6B attention shape 16/8/128, bs 256,
768-block pool, max_num_batched_tokens 16384, max_num_seqs 512) through
``EngineReplay``, the step loop the benchmark times: the native scheduler,
eager kv_store + attn_prefill_varlen per layer for prefill steps, and for
decode steps one packed metadata copy plus one replay of the 28-layer graph
of attn_decode_paged_append ("nano-vLLM-1", ModelRunner "7. 性能优化":
decode runs as a captured graph; Scheduler "2. prefill 的 schedule" /
"3. decode 的 schedule").  Every layer gets its own q/k/v.

The oracle follows layers 0 and 27: it replays every store (the caches must
match bit for bit at the end), checks attention on every prefill step (a
seeded sample of rows) and, on a seeded 6% of the decode steps plus the
first ones, every sequence of the step."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import engine_trace as E
from paged_kv_cache_125_gb300.engine_replay import EngineReplay

from parity import BF16_NAN, assert_attn_close, u16

pytestmark = pytest.mark.gpu

LAYERS, HQ, HKV, D, BS, NB = 28, 16, 8, 128, 256, 768
CHECK_LAYERS = (0, 27)


def test_config5_trace_replay_through_the_benchmark_path():
    dev = torch.device("cuda")
    eng = EngineReplay(E.make_requests(256, (100, 1024), (100, 1024)), LAYERS, HQ, HKV, D, BS, NB,
                       512, 16384, dev)
    ora = {l: (np.full((NB, BS, HKV, D), BF16_NAN, np.uint16), np.full((NB, BS, HKV, D), BF16_NAN, np.uint16))
           for l in CHECK_LAYERS}
    scale = D ** -0.5
    gen = torch.Generator(device=dev).manual_seed(11)
    rng = np.random.default_rng(5)
    checked = {"prefill": 0, "decode": 0}
    steps = decode_steps = 0
    while not eng.done():
        st = eng.schedule()
        m, n = st.meta, st.num_new
        if st.is_prefill:
            q = torch.randn((LAYERS, n, HQ, D), generator=gen, device=dev).to(torch.bfloat16)
            k = torch.randn((LAYERS, n, HKV, D), generator=gen, device=dev).to(torch.bfloat16)
            v = torch.randn((LAYERS, n, HKV, D), generator=gen, device=dev).to(torch.bfloat16)
            outs = eng.launch(st, q, k, v)
            rows = np.sort(rng.choice(n, size=min(n, 160), replace=False))
            for l in CHECK_LAYERS:
                okc, ovc = ora[l]
                ql, kl, vl = q[l].cpu(), k[l].cpu(), v[l].cpu()
                oracle.kv_store(kl, vl, m.slot_mapping, okc, ovc)
                if m.block_tables is None:
                    ref = oracle.prefill(ql, m.cu_seqlens_q, m.cu_seqlens_k, HQ, HKV, scale, k=kl, v=vl,
                                         rows=rows)
                else:
                    ref = oracle.prefill(ql, m.cu_seqlens_q, m.cu_seqlens_k, HQ, HKV, scale, k_cache=okc,
                                         v_cache=ovc, block_tables=m.block_tables, rows=rows)
                assert_attn_close(outs[l], ref, f"step {steps} layer {l} (prefill)", rows)
            checked["prefill"] += 1
        else:
            q, k, v = eng.decode_inputs(st)
            q.copy_(torch.randn(q.shape, generator=gen, device=dev))
            k.copy_(torch.randn(k.shape, generator=gen, device=dev))
            v.copy_(torch.randn(v.shape, generator=gen, device=dev))
            check = decode_steps < 2 or rng.random() < 0.06
            out = eng.launch(st)
            for l in CHECK_LAYERS:
                okc, ovc = ora[l]
                oracle.kv_store(k[l].cpu(), v[l].cpu(), m.slot_mapping, okc, ovc)
                if check:
                    ref = oracle.decode(q[l].cpu(), okc, ovc, m.block_tables, m.context_lens, HQ, HKV, scale)
                    assert_attn_close(out[l], ref, f"step {steps} layer {l} (decode)")
            checked["decode"] += check
            decode_steps += 1
        eng.commit(st, [E.synthetic_token(i, steps) for i in st.seq_ids])
        steps += 1
    torch.cuda.synchronize()
    assert kvp.device_status() == 0
    assert steps > 1000 and eng.num_preemptions > 0
    prefill_steps = steps - decode_steps
    assert checked["prefill"] == prefill_steps
    assert checked["decode"] >= 0.05 * decode_steps, checked
    for l in CHECK_LAYERS:
        okc, ovc = ora[l]
        kc, vc = eng.cache(l)
        assert np.array_equal(u16(kc), okc), f"layer {l} K cache"
        assert np.array_equal(u16(vc), ovc), f"layer {l} V cache"
