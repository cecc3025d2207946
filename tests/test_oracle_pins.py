"""Pins for the CPU oracle: checks against things other than the oracle itself.

* brute force: textbook contiguous attention, softmax(Q K^T * scale + causal
  mask) V, written with numpy matmul and scipy's softmax, and torch's fp64
  scaled_dot_product_attention (page 3, "KV-Cache … 是什么？");
* closed forms: q = 0 gives uniform weights, so row i is the mean of the
  values it sees; a row that sees one key returns that key's value exactly;
* invariances the pages state or imply: relabelling physical blocks changes
  nothing (paging, page 3 "PageAttention"); a prefix-cached suffix prefill
  equals the same rows of a full prefill, and decoding token L-1 equals row L-1
  of a causal prefill (causal invariance, page 3 "KV-Cache … 是什么？");
* store-then-gather returns the stored bits, and the pages' paging examples;
* copy on write (page 3, "场景优化1：Parallel Memory Shared"): two sampled
  sequences share a partly filled prompt block; after the copy each appends
  its own token and reads back exactly prompt + own token, in every layer.
"""
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_kv_cache_125_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "paging_examples.json")


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.float().double().numpy()


def brute_prefill(q, k_full, v_full, q_lens, k_lens, hq, hkv, scale):
    """Contiguous textbook attention per sequence; k_full/v_full are the
    sequences' full keys concatenated [sum k, Hkv, d]."""
    qd, kd, vd = bf16_np(q), bf16_np(k_full), bf16_np(v_full)
    out = np.zeros(qd.shape)
    g = hq // hkv
    cq = ck = 0
    for ql, kl in zip(q_lens, k_lens):
        c = kl - ql
        for h in range(hq):
            Q = qd[cq:cq + ql, h, :]
            K = kd[ck:ck + kl, h // g, :]
            V = vd[ck:ck + kl, h // g, :]
            S = Q @ K.T * scale
            i = np.arange(ql)[:, None]
            j = np.arange(kl)[None, :]
            S = np.where(j <= c + i, S, -np.inf)
            out[cq:cq + ql, h, :] = scipy.special.softmax(S, axis=1) @ V
        cq += ql
        ck += kl
    return out


def empty_pool(nb, bs, hkv, d):
    nan = np.uint16(0x7FC0)  # bf16 quiet NaN
    return np.full((nb, bs, hkv, d), nan, np.uint16), np.full((nb, bs, hkv, d), nan, np.uint16)


def random_paged_case(seed, seq_lens, cached_blocks, hq, hkv, d, bs, nb):
    """Full K/V of every sequence stored into a NaN pool through random block
    tables; returns what the paged prefill needs plus the contiguous copy."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(nb, generator=g).tolist()
    tables, at = [], 0
    for L in seq_lens:
        n = W.num_blocks_for(L, bs)
        tables.append(perm[at:at + n])
        at += n
    k_full = torch.randn((sum(seq_lens), hkv, d), generator=g).to(torch.bfloat16)
    v_full = torch.randn((sum(seq_lens), hkv, d), generator=g).to(torch.bfloat16)
    slots = []
    for bt, L in zip(tables, seq_lens):
        slots += W.slots_of_positions(bt, range(L), bs)
    kc, vc = empty_pool(nb, bs, hkv, d)
    oracle.kv_store(k_full, v_full, torch.tensor(slots, dtype=torch.int32), kc, vc)
    cached = [c * bs for c in cached_blocks]
    meta = W.prefill_metadata(seq_lens, cached, tables, bs)
    q = torch.randn((int(meta.cu_seqlens_q[-1]), hq, d), generator=g).to(torch.bfloat16)
    return dict(q=q, k_full=k_full, v_full=v_full, kc=kc, vc=vc, tables=tables, meta=meta,
                q_lens=[L - c for L, c in zip(seq_lens, cached)], k_lens=list(seq_lens),
                bt=W.prepare_block_tables(tables))


# --------------------------------------------------------------------------- store / gather

def test_store_then_gather_roundtrips_bits():
    g = torch.Generator().manual_seed(11)
    nb, bs, hkv, d = 40, 16, 2, 64
    lens = [37, 100, 16, 1]
    perm = torch.randperm(nb, generator=g).tolist()
    tables, at = [], 0
    for L in lens:
        n = W.num_blocks_for(L, bs)
        tables.append(perm[at:at + n])
        at += n
    k = torch.randn((sum(lens), hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((sum(lens), hkv, d), generator=g).to(torch.bfloat16)
    slots = [s for bt, L in zip(tables, lens) for s in W.slots_of_positions(bt, range(L), bs)]
    kc, vc = empty_pool(nb, bs, hkv, d)
    oracle.kv_store(k, v, torch.tensor(slots, dtype=torch.int32), kc, vc)
    ku = k.view(torch.int16).numpy().view(np.uint16)
    vu = v.view(torch.int16).numpy().view(np.uint16)
    at = 0
    for bt, L in zip(tables, lens):
        assert np.array_equal(oracle.gather(kc, bt, L), ku[at:at + L])
        assert np.array_equal(oracle.gather(vc, bt, L), vu[at:at + L])
        at += L
    # every slot not written is still the NaN poison
    written = np.zeros(nb * bs, bool)
    written[slots] = True
    assert np.all(kc.reshape(nb * bs, -1)[~written] == 0x7FC0)


def test_store_skips_negative_slots():
    nb, bs, hkv, d = 4, 16, 1, 64
    k = torch.randn((3, hkv, d)).to(torch.bfloat16)
    kc, vc = empty_pool(nb, bs, hkv, d)
    before = kc.copy()
    oracle.kv_store(k, k, torch.tensor([-1, 5, -1], dtype=torch.int32), kc, vc)
    changed = np.argwhere(np.any(kc.reshape(nb * bs, -1) != before.reshape(nb * bs, -1), axis=1)).ravel()
    assert changed.tolist() == [5]


def test_store_rejects_slot_past_pool():
    kc, vc = empty_pool(2, 16, 1, 64)
    k = torch.zeros((1, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(oracle.OracleError):
        oracle.kv_store(k, k, torch.tensor([32], dtype=torch.int32), kc, vc)


def test_pages_paging_examples():
    ex = json.load(open(GOLDEN))
    lk = ex["block_table_lookup"]
    bs = 4
    nb = 16
    kc, vc = empty_pool(nb, bs, 1, 64)
    # mark every physical block with its own id in dim 0, then gather logical blocks
    for blk in range(nb):
        kc[blk, :, 0, 0] = blk
    got = oracle.gather(kc, lk["block_table"], bs * len(lk["block_table"]))
    for logical, physical in lk["logical_to_physical"]:
        assert np.all(got[logical * bs:(logical + 1) * bs, 0, 0] == physical)

    fig = ex["figure_bs4"]
    meta = W.prefill_metadata([fig["prompt_len"]], [0], [fig["block_table"]], fig["block_size"])
    assert meta.slot_mapping.tolist() == fig["prefill_slots"]
    assert meta.block_tables is None  # nothing cached -> no block tables (prefill path)
    dm = W.decode_metadata([fig["prompt_len"] + 1], [fig["block_table"]], fig["block_size"])
    assert dm.slot_mapping.tolist() == [fig["eighth_token_slot"]]
    assert dm.context_lens.tolist() == [8] and dm.positions.tolist() == [7]
    assert W.num_blocks_for(fig["prompt_len"] + 2, fig["block_size"]) == 3  # ninth token: new block

    sf = ex["slot_formula"]
    assert W.slots_of_positions(sf["block_table"], sf["positions"], sf["block_size"]) == sf["slots"]


# --------------------------------------------------------------------------- attention

@pytest.mark.parametrize("hq,hkv,d", [(2, 1, 64), (4, 2, 32), (8, 2, 128)])
def test_prefill_matches_brute_force_packed(hq, hkv, d):
    g = torch.Generator().manual_seed(hq * 100 + d)
    lens = [1, 9, 33]
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    q = torch.randn((sum(lens), hq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((sum(lens), hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((sum(lens), hkv, d), generator=g).to(torch.bfloat16)
    scale = 1 / np.sqrt(d)
    got = oracle.prefill(q, cu, cu, hq, hkv, scale, k=k, v=v)
    want = brute_prefill(q, k, v, lens, lens, hq, hkv, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_prefill_matches_torch_sdpa_fp64():
    g = torch.Generator().manual_seed(5)
    L, hq, hkv, d = 45, 6, 3, 16
    q = torch.randn((L, hq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((L, hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((L, hkv, d), generator=g).to(torch.bfloat16)
    cu = torch.tensor([0, L], dtype=torch.int32)
    got = oracle.prefill(q, cu, cu, hq, hkv, 1 / np.sqrt(d), k=k, v=v)
    rep = hq // hkv
    Q = q.double().permute(1, 0, 2)
    K = k.double().repeat_interleave(rep, dim=1).permute(1, 0, 2)
    V = v.double().repeat_interleave(rep, dim=1).permute(1, 0, 2)
    want = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True)
    np.testing.assert_allclose(got, want.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("bs", [16, 32])
def test_prefill_paged_prefix_matches_brute_force(bs):
    c = random_paged_case(7 + bs, [70, 129, 40], [2, 3, 0], 4, 2, 64, bs, 64)
    m = c["meta"]
    assert m.block_tables is not None
    got = oracle.prefill(c["q"], m.cu_seqlens_q, m.cu_seqlens_k, 4, 2, 0.125,
                         k_cache=c["kc"], v_cache=c["vc"], block_tables=m.block_tables)
    want = brute_prefill(c["q"], c["k_full"], c["v_full"], c["q_lens"], c["k_lens"], 4, 2, 0.125)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_uniform_weights_closed_form():
    """q = 0 makes every visible score 0: row i (position c+i) is the mean of
    values 0..c+i of its kv head.  Pins the inclusive diagonal, the prefix
    offset and the GQA head mapping."""
    bs, hq, hkv, d = 16, 4, 2, 8
    c = random_paged_case(3, [50], [2], hq, hkv, d, bs, 16)
    q = torch.zeros_like(c["q"])
    m = c["meta"]
    got = oracle.prefill(q, m.cu_seqlens_q, m.cu_seqlens_k, hq, hkv, 1.0,
                         k_cache=c["kc"], v_cache=c["vc"], block_tables=m.block_tables)
    vf = bf16_np(c["v_full"])
    cached = 32
    for i in range(50 - cached):
        for h in range(hq):
            want = vf[:cached + i + 1, h // 2, :].mean(axis=0)
            np.testing.assert_allclose(got[i, h], want, rtol=1e-13, atol=1e-14)


def test_single_visible_key_returns_its_value_exactly():
    g = torch.Generator().manual_seed(1)
    q = torch.randn((5, 2, 64), generator=g).to(torch.bfloat16)
    k = torch.randn((5, 1, 64), generator=g).to(torch.bfloat16)
    v = torch.randn((5, 1, 64), generator=g).to(torch.bfloat16)
    cu = torch.tensor([0, 5], dtype=torch.int32)
    got = oracle.prefill(q, cu, cu, 2, 1, 0.125, k=k, v=v)
    assert np.array_equal(got[0, 0], bf16_np(v)[0, 0]) and np.array_equal(got[0, 1], bf16_np(v)[0, 0])


def test_peaked_softmax_selects_best_key():
    g = torch.Generator().manual_seed(2)
    L, d = 20, 64
    q = torch.randn((L, 1, d), generator=g).to(torch.bfloat16)
    k = torch.randn((L, 1, d), generator=g).to(torch.bfloat16)
    v = torch.randn((L, 1, d), generator=g).to(torch.bfloat16)
    cu = torch.tensor([0, L], dtype=torch.int32)
    got = oracle.prefill(q, cu, cu, 1, 1, 1e4, k=k, v=v)
    qd, kd, vd = bf16_np(q), bf16_np(k), bf16_np(v)
    for i in range(L):
        best = int(np.argmax(kd[:i + 1, 0] @ qd[i, 0]))
        np.testing.assert_allclose(got[i, 0], vd[best, 0], atol=1e-9)


def test_block_relabelling_invariance():
    """Moving every physical block to another id (and its data with it) leaves
    prefill and decode outputs bit-identical."""
    bs, nb, hq, hkv, d = 16, 48, 4, 2, 64
    c = random_paged_case(9, [90, 33], [1, 2], hq, hkv, d, bs, nb)
    m = c["meta"]
    base = oracle.prefill(c["q"], m.cu_seqlens_q, m.cu_seqlens_k, hq, hkv, 0.125,
                          k_cache=c["kc"], v_cache=c["vc"], block_tables=m.block_tables)
    relabel = torch.randperm(nb, generator=torch.Generator().manual_seed(4)).numpy()
    kc2, vc2 = np.empty_like(c["kc"]), np.empty_like(c["vc"])
    kc2[relabel] = c["kc"]
    vc2[relabel] = c["vc"]
    bt = m.block_tables.numpy()
    bt2 = np.where(bt >= 0, relabel[np.maximum(bt, 0)], -1).astype(np.int32)
    moved = oracle.prefill(c["q"], m.cu_seqlens_q, m.cu_seqlens_k, hq, hkv, 0.125,
                           k_cache=kc2, v_cache=vc2, block_tables=bt2)
    assert np.array_equal(base, moved)
    qd = torch.randn((2, hq, d)).to(torch.bfloat16)
    ctx = torch.tensor([90, 33], dtype=torch.int32)
    d1 = oracle.decode(qd, c["kc"], c["vc"], bt, ctx, hq, hkv, 0.125)
    d2 = oracle.decode(qd, kc2, vc2, bt2, ctx, hq, hkv, 0.125)
    assert np.array_equal(d1, d2)


def test_prefix_cached_suffix_equals_full_prefill_rows():
    bs, hq, hkv, d = 16, 4, 2, 32
    full = random_paged_case(21, [100], [0], hq, hkv, d, bs, 16)
    fm = full["meta"]
    # the same pool/tables, now with 3 blocks (48 tokens) already cached
    pm = W.prefill_metadata([100], [48], full["tables"], bs)
    a = oracle.prefill(full["q"], fm.cu_seqlens_q, fm.cu_seqlens_k, hq, hkv, 0.2,
                       k_cache=full["kc"], v_cache=full["vc"], block_tables=full["bt"])
    b = oracle.prefill(full["q"][48:], pm.cu_seqlens_q, pm.cu_seqlens_k, hq, hkv, 0.2,
                       k_cache=full["kc"], v_cache=full["vc"], block_tables=pm.block_tables)
    assert np.array_equal(a[48:], b)


def test_decode_equals_last_prefill_row():
    bs, hq, hkv, d = 16, 4, 2, 64
    c = random_paged_case(31, [77, 16, 1], [0, 0, 0], hq, hkv, d, bs, 32)
    cu = c["meta"].cu_seqlens_q
    pre = oracle.prefill(c["q"], cu, cu, hq, hkv, 0.125, k_cache=c["kc"], v_cache=c["vc"],
                         block_tables=c["bt"])
    last_rows = (cu[1:] - 1).long()
    dec = oracle.decode(c["q"][last_rows], c["kc"], c["vc"], c["bt"],
                        torch.tensor([77, 16, 1], dtype=torch.int32), hq, hkv, 0.125)
    np.testing.assert_allclose(dec, pre[last_rows.numpy()], rtol=0, atol=1e-15)


def test_decode_zero_context_is_zero_and_reads_nothing():
    kc, vc = empty_pool(4, 16, 1, 64)  # all NaN: any read would poison the result
    q = torch.randn((2, 2, 64)).to(torch.bfloat16)
    bt = np.full((2, 1), -1, np.int32)
    out = oracle.decode(q, kc, vc, bt, torch.tensor([0, 0], dtype=torch.int32), 2, 1, 0.125)
    assert np.all(out == 0)


def test_decode_subset_matches_full():
    c = random_paged_case(41, [30, 60, 90], [0, 0, 0], 4, 2, 64, 16, 32)
    q = torch.randn((3, 4, 64)).to(torch.bfloat16)
    ctx = torch.tensor([30, 60, 90], dtype=torch.int32)
    full = oracle.decode(q, c["kc"], c["vc"], c["bt"], ctx, 4, 2, 0.125)
    sub = oracle.decode(q, c["kc"], c["vc"], c["bt"], ctx, 4, 2, 0.125, seqs=[2, 0])
    assert np.array_equal(sub[[0, 2]], full[[0, 2]]) and np.all(sub[1] == 0)


def test_copy_on_write_parallel_sampling():
    """Page 3's parallel-sampling example: sequences A1 and A2 come from one
    prompt and share its physical blocks; the last one is partly filled.  A1
    must append, sees a reference count of 2, gets a new block holding a copy
    of the shared one, and writes its token there; A2 then appends into the
    original block.  Checked in each of 3 layers (6 planes) through the
    store and gather of the pages' slot formula: each sequence reads back
    exactly the prompt rows followed by its own new row."""
    g = torch.Generator().manual_seed(21)
    layers, nb, bs, hkv, d = 3, 12, 4, 2, 8
    prompt_len = 6                      # blocks: one full, one with 2 of 4 slots
    table = [7, 2]                      # shared physical blocks of the prompt
    cache = np.full((2, layers, nb, bs, hkv, d), 0x7FC0, dtype=np.uint16)
    prompt = torch.randn((2, layers, prompt_len, hkv, d), generator=g).to(torch.bfloat16)
    slots = torch.tensor(W.slots_of_positions(table, range(prompt_len), bs), dtype=torch.int32)
    for layer in range(layers):
        kc, vc = cache[0, layer], cache[1, layer]
        oracle.kv_store(prompt[0, layer], prompt[1, layer], slots, kc, vc)
    new_block = 9                       # free block given to A1
    oracle.copy_blocks(cache, [[table[-1], new_block]])
    t1 = [table[0], new_block]
    t2 = list(table)
    tok = torch.randn((2, 2, layers, 1, hkv, d), generator=g).to(torch.bfloat16)  # [seq, k/v, layer]
    pos = prompt_len                    # the appended token's position
    for layer in range(layers):
        for seq, bt in ((0, t1), (1, t2)):
            s_ = torch.tensor(W.slots_of_positions(bt, [pos], bs), dtype=torch.int32)
            oracle.kv_store(tok[seq, 0, layer], tok[seq, 1, layer], s_, cache[0, layer], cache[1, layer])
    u = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    for layer in range(layers):
        for kv in range(2):
            for seq, bt in ((0, t1), (1, t2)):
                got = oracle.gather(cache[kv, layer], bt, prompt_len + 1)
                want = np.concatenate([u(prompt[kv, layer]), u(tok[seq, kv, layer])])
                assert np.array_equal(got, want), (layer, kv, seq)
    # blocks nobody wrote keep the poison
    untouched = [b for b in range(nb) if b not in (7, 2, 9)]
    assert np.all(cache[:, :, untouched] == 0x7FC0)


def test_copy_blocks_leaves_everything_but_destinations():
    """Several pairs over 4 planes: every destination block equals its
    source's previous content; every other block (sources included) keeps
    its bits."""
    rng = np.random.default_rng(5)
    cache = rng.integers(0, 1 << 16, size=(4, 20, 3, 2, 8), dtype=np.uint16)
    before = cache.copy()
    pairs = [[3, 11], [3, 12], [0, 19], [7, 5]]
    oracle.copy_blocks(cache, pairs)
    dsts = {d_ for _, d_ in pairs}
    for s_, d_ in pairs:
        assert np.array_equal(cache[:, d_], before[:, s_])
    for b in range(20):
        if b not in dsts:
            assert np.array_equal(cache[:, b], before[:, b])


def test_copy_blocks_rejects_out_of_range():
    cache = np.zeros((2, 4, 2, 1, 8), dtype=np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(cache, [[0, 4]])
