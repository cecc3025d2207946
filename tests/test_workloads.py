"""Host-side metadata builders and seeded workloads (no GPU)."""
import torch

from paged_kv_cache_125_gb300 import workloads as W


def test_prefill_metadata_matches_per_position_slots():
    bs = 16
    tables = [[3, 9, 1], [7], [2, 5, 11, 0]]
    lens, cached = [40, 16, 50], [16, 0, 48]
    m = W.prefill_metadata(lens, cached, tables, bs)
    want = []
    for bt, L, c in zip(tables, lens, cached):
        want += W.slots_of_positions(bt, range(c, L), bs)
    assert m.slot_mapping.tolist() == want
    assert m.cu_seqlens_q.tolist() == [0, 24, 40, 42]
    assert m.cu_seqlens_k.tolist() == [0, 40, 56, 106]
    assert (m.max_seqlen_q, m.max_seqlen_k) == (24, 50)
    assert m.positions.tolist() == list(range(16, 40)) + list(range(16)) + [48, 49]
    assert m.block_tables.tolist() == [[3, 9, 1, -1], [7, -1, -1, -1], [2, 5, 11, 0]]


def test_no_block_tables_without_prefix_hit():
    m = W.prefill_metadata([5, 20], [0, 0], [[1], [4, 6]], 16)
    assert m.block_tables is None


def test_decode_metadata_last_slot():
    bs = 16
    m = W.decode_metadata([17, 32, 1], [[4, 8], [1, 2], [9]], bs)
    assert m.slot_mapping.tolist() == [8 * 16 + 0, 2 * 16 + 15, 9 * 16]
    assert m.context_lens.tolist() == [17, 32, 1] and m.positions.tolist() == [16, 31, 0]
    assert m.max_context_len == 32


def test_tiny_workload_shape():
    w = W.config1_tiny()
    assert len(w.steps) == 5 and w.steps[0].is_prefill
    pre = w.steps[0].attn
    assert pre.meta.cu_seqlens_q.tolist() == [0, 17, 17 + 284]
    assert pre.meta.cu_seqlens_k.tolist() == [0, 17, 317]
    assert pre.meta.block_tables is not None
    assert w.setup[0].slot_mapping.numel() == 16
    ctx = [s.attn.meta.context_lens.tolist() for s in w.steps[1:]]
    assert ctx == [[18, 301], [19, 302], [20, 303], [21, 304]]
    # all slots written over the whole workload are distinct
    allslots = torch.cat([w.setup[0].slot_mapping] + [s.store.slot_mapping for s in w.steps])
    assert allslots.unique().numel() == allslots.numel()


def test_config3_caps_cached_blocks():
    w = W.config3_prefill()
    m = w.steps[0].attn.meta
    ql = (m.cu_seqlens_q[1:] - m.cu_seqlens_q[:-1]).tolist()
    kl = (m.cu_seqlens_k[1:] - m.cu_seqlens_k[:-1]).tolist()
    assert all(q >= 1 for q in ql)
    assert all((k - q) % 256 == 0 and (k - q) // 256 in (0, 1, 2) for q, k in zip(ql, kl))
    assert all(256 <= k <= 2048 for k in kl) and sum(kl) <= 16384


def test_decode_workload_history_excludes_new_token():
    w = W.decode_workload("t", [5, 20], 2, 1, 64, 16, 8)
    assert w.history_slots.numel() == 4 + 19
    st = w.steps[0].store
    assert not set(st.slot_mapping.tolist()) & set(w.history_slots.tolist())
