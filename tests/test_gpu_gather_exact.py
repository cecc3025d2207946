"""Bit-exact pin of the block-table gather inside the paged attention kernels.

The gather (logical token p of sequence b lives at slot
block_tables[b][p // bs] * bs + p % bs: "nano-vLLM-1", BlockManager
"3. 核心方法一：分配 (allocate)"; "【nano-vllm 学习】04 …", "代码分析",
block_table [5, 12, 3]) is folded into the K/V loads of the decode and prefill
kernels, so an ordinary parity test sees it only through the attention
tolerance.  Here every output row is made to equal one V row exactly:

* query head j of a kv group is c * H[1 + j], a row of a +-1 Hadamard matrix
  (c = 8), and for every (sequence, kv head, j) one key position p_j holds
  K = c * H[1 + j].  That key scores c^2 * d for head j; the keys of the other
  heads' targets score 0 (Hadamard rows are orthogonal) and the N(0,1) keys
  score about c * N(0, 1) * sqrt(d).  In base-2 units after the 1/sqrt(d)
  scale the gap exceeds 500, so every other softmax weight underflows to 0 in
  fp32 (and to below 1e-200 in the oracle's fp64): the output is exactly
  V[p_j] of that kv head.
* Targets cover every in-block offset (bs 16) or a spread of them (bs 256),
  many block ids of shuffled block tables, both slots of the prefill kernel's
  K/V rings and every stage of the decode ring.

The expected bits come from the oracle's gather of the V cache; the oracle's
own attention output (rounded to bf16) is checked to equal them too.  A
prefill row that sits before its target sees only random keys; those rows are
checked against the oracle within the attention tolerance."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import workloads as W

from parity import assert_attn_close, gpu_pool, oracle_pool, u16

pytestmark = pytest.mark.gpu

C = 8.0


def hadamard(n: int) -> np.ndarray:
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def bf16_bits_of_f64(x: np.ndarray) -> np.ndarray:
    return u16(torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16))


def pick_targets(lens, hkv, G, bs, seed):
    """-> {(b, g, j): position}, distinct positions per (b, g); offsets within
    a block cycle through 0..bs-1 over the targets, block ids are random."""
    rng = np.random.default_rng(seed)
    out, t = {}, 0
    for b, L in enumerate(lens):
        nblk = W.num_blocks_for(L, bs)
        assert L == 1 or L >= G
        for g in range(hkv):
            if L == 1:  # a single visible key: every head's output is V[0]
                out.update({(b, g, j): 0 for j in range(G)})
                continue
            used = set()
            for j in range(G):
                lb = int(rng.integers(0, nblk))
                p = min(lb * bs + (t * 7) % bs, L - 1)
                while p in used:
                    p = (p + 1) % L
                used.add(p)
                out[(b, g, j)] = p
                t += 1
    return out


def peak_queries(q, hkv, G, d):
    """q[:, g*G + j] = C * H[1 + j] for every row."""
    h = hadamard(d)
    pat = torch.tensor(C * h[1:1 + G], dtype=torch.float32).to(torch.bfloat16)
    q.copy_(pat.repeat(hkv, 1).unsqueeze(0).expand_as(q))


def key_pattern(j, d):
    return torch.tensor(C * hadamard(d)[1 + j], dtype=torch.float32).to(torch.bfloat16)


def expected_rows(vc_np, tables, lens, targets, hq, hkv, G, d):
    """-> uint16 [B, Hq, d]: V[p_j] of each head's kv head, read by the oracle's gather."""
    exp = np.zeros((len(lens), hq, d), dtype=np.uint16)
    for b, L in enumerate(lens):
        rows = oracle.gather(vc_np, tables[b], L)
        for g in range(hkv):
            for j in range(G):
                exp[b, g * G + j] = rows[targets[(b, g, j)], g]
    return exp


# --------------------------------------------------------------------------- decode

def decode_case(name, lens, hq, hkv, d, bs, nb, seed):
    w = W.decode_workload(name, lens, hq, hkv, d, bs, nb)
    G = hq // hkv
    targets = pick_targets(lens, hkv, G, bs, seed)
    st, a = w.steps[0].store, w.steps[0].attn
    hist_k = w.history_k.clone()
    base = np.cumsum([0] + [L - 1 for L in lens])
    for (b, g, j), p in targets.items():
        if lens[b] == 1 and j > 0:
            continue  # the one key carries head 0's pattern; the others score 0 on it
        if p == lens[b] - 1:
            st.k[b, g] = key_pattern(j, d)
        else:
            hist_k[base[b] + p, g] = key_pattern(j, d)
    w.history_k = hist_k
    peak_queries(a.q, hkv, G, d)
    return w, targets


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_store"])
@pytest.mark.parametrize("hq,hkv,d,bs,lens,nb", [
    (16, 8, 128, 16, [1, 16, 17, 33, 250, 511, 1000, 2047] * 4, 2048),
    (32, 8, 128, 256, [300, 1, 4096, 257, 2000, 255, 3333, 700], 256),
    (16, 8, 128, 256, [4096 * 4, 5, 512], 96),       # one sequence crosses many CTAs
    (8, 2, 64, 16, [40, 600, 17, 3000], 300),
])
def test_decode_gather_bit_exact(hq, hkv, d, bs, lens, nb, fused):
    w, targets = decode_case(f"gather_dec_{hq}_{d}_{bs}", lens, hq, hkv, d, bs, nb, seed=len(lens) + bs)
    G = hq // hkv
    step = w.steps[0]
    m = step.attn.meta
    kc, vc = gpu_pool(w)
    if fused:
        out = kvp.attn_decode_paged_append(step.attn.q.cuda(), step.store.k.cuda(), step.store.v.cuda(),
                                           m.slot_mapping.cuda(), kc, vc, m.block_tables.cuda(),
                                           m.context_lens.cuda(), m.max_context_len, softmax_scale=w.scale)
    else:
        kvp.kv_store(step.store.k.cuda(), step.store.v.cuda(), m.slot_mapping.cuda(), kc, vc)
        out = kvp.attn_decode_paged(step.attn.q.cuda(), kc, vc, m.block_tables.cuda(), m.context_lens.cuda(),
                                    m.max_context_len, softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert kvp.device_status() == 0
    # oracle side: store, then gather the expected V rows
    kr, vr = oracle_pool(w)
    oracle.kv_store(step.store.k, step.store.v, m.slot_mapping, kr, vr)
    tables = [m.block_tables[b].tolist() for b in range(len(lens))]
    exp = expected_rows(vr, tables, lens, targets, hq, hkv, G, d)
    ref = oracle.decode(step.attn.q, kr, vr, m.block_tables, m.context_lens, hq, hkv, w.scale)
    assert np.array_equal(bf16_bits_of_f64(ref), exp), "the construction is not exact in the oracle"
    got = u16(out)
    bad = np.argwhere((got != exp).any(axis=2))
    assert bad.size == 0, f"{len(bad)} (seq, head) rows differ, first {bad[:4].tolist()}"


# --------------------------------------------------------------------------- prefill

@pytest.mark.parametrize("hq,hkv,d,bs,lens,cached_blocks,nb", [
    (32, 8, 128, 256, [256, 2048, 700, 1500, 257, 1024], [1, 2, 0, 1, 1, 0], 64),
    (16, 8, 128, 16, [600, 130, 2000, 48, 1000], [3, 8, 0, 1, 20], 512),
    (16, 8, 128, 256, [3000, 513], [2, 1], 24),
    (8, 2, 64, 16, [300, 999], [2, 17], 128),
])
def test_prefill_gather_bit_exact(hq, hkv, d, bs, lens, cached_blocks, nb):
    w = W.prefill_workload(f"gather_pf_{hq}_{d}_{bs}", lens, cached_blocks, hq, hkv, d, bs, nb)
    G = hq // hkv
    step = w.steps[0]
    m = step.attn.meta
    cached = [c * bs for c in cached_blocks]
    targets = pick_targets(lens, hkv, G, bs, seed=sum(lens))
    pre_base = np.cumsum([0] + cached)
    cq = m.cu_seqlens_q.tolist()
    for (b, g, j), p in targets.items():
        if p < cached[b]:
            w.setup[0].k[pre_base[b] + p, g] = key_pattern(j, d)
        else:
            step.store.k[cq[b] + p - cached[b], g] = key_pattern(j, d)
    peak_queries(step.attn.q, hkv, G, d)
    assert m.block_tables is not None

    kc, vc = gpu_pool(w)
    for s in w.setup:
        kvp.kv_store(s.k.cuda(), s.v.cuda(), s.slot_mapping.cuda(), kc, vc)
    kvp.kv_store(step.store.k.cuda(), step.store.v.cuda(), m.slot_mapping.cuda(), kc, vc)
    out = kvp.attn_prefill_varlen(step.attn.q.cuda(), m.cu_seqlens_q.cuda(), m.cu_seqlens_k.cuda(),
                                  m.max_seqlen_q, m.max_seqlen_k, k_cache=kc, v_cache=vc,
                                  block_tables=m.block_tables.cuda(), num_kv_heads=hkv,
                                  softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert kvp.device_status() == 0

    kr, vr = oracle_pool(w)
    for s in w.setup:
        oracle.kv_store(s.k, s.v, s.slot_mapping, kr, vr)
    oracle.kv_store(step.store.k, step.store.v, m.slot_mapping, kr, vr)
    ref = oracle.prefill(step.attn.q, m.cu_seqlens_q, m.cu_seqlens_k, hq, hkv, w.scale,
                         k_cache=kr, v_cache=vr, block_tables=m.block_tables)
    tables = [m.block_tables[b].tolist() for b in range(len(lens))]
    got = u16(out)
    ref_bits = bf16_bits_of_f64(ref)
    exact = np.zeros(got.shape[:2], dtype=bool)
    n_exact = 0
    for b, L in enumerate(lens):
        rows = oracle.gather(vr, tables[b], L)
        for i in range(L - cached[b]):
            pos = cached[b] + i
            for g in range(hkv):
                for j in range(G):
                    p = targets[(b, g, j)]
                    if p <= pos:
                        r, h = cq[b] + i, g * G + j
                        exact[r, h] = True
                        assert np.array_equal(ref_bits[r, h], rows[p, g]), "oracle not exact"
                        if not np.array_equal(got[r, h], rows[p, g]):
                            raise AssertionError(f"seq {b} row {i} (position {pos}) head {h}: "
                                                 f"differs from V[{p}] of kv head {g}")
                        n_exact += 1
    assert n_exact > 0.5 * exact.size
    # rows before their target: ordinary attention over random keys
    assert_attn_close(out, ref, "rows before their target", mask=~exact)
