"""The engine-step trace generator (scheduler / block-manager replica of the
pages' policy): invariants checked at every step, on CPU."""
import pytest
import torch

from paged_kv_cache_125_gb300 import engine_trace as E
from paged_kv_cache_125_gb300 import workloads as W


def _check_step(st, sched, bs):
    pool = sched.pool
    nb = pool.num_blocks
    free, used = set(pool.free_queue), pool.in_use()
    assert not (free & used) and len(free) + len(used) == nb, "free and used must partition the pool"
    assert pool.num_free == len(free), "free queue holds no duplicates"
    # reference counts equal the number of tables holding each block
    holders = {}
    for seq in sched.running:
        for b in seq.table:
            holders[b] = holders.get(b, 0) + 1
    for b in range(nb):
        assert pool.refs[b] == holders.get(b, 0)
    m = st.meta
    slots = m.slot_mapping.tolist()
    assert len(set(slots)) == len(slots), "a slot is written twice in one step"
    seqs = {s.rid: s for s in sched.running}
    if st.is_prefill:
        cq, ck = m.cu_seqlens_q.tolist(), m.cu_seqlens_k.tolist()
        at = 0
        for i, sid in enumerate(st.seq_ids):
            s = seqs[sid]
            assert ck[i + 1] - ck[i] == len(s)
            assert ck[i + 1] - ck[i] - (cq[i + 1] - cq[i]) == s.cached
            want = W.slots_of_positions(s.table, range(s.cached, len(s)), bs)
            assert slots[at:at + len(want)] == want
            at += len(want)
        assert at == len(slots)
        assert sum(len(s) for s in (seqs[i] for i in st.seq_ids)) <= sched.max_num_batched_tokens
    else:
        for i, sid in enumerate(st.seq_ids):
            s = seqs[sid]
            assert m.context_lens[i] == len(s)
            assert slots[i] == W.slots_of_positions(s.table, [len(s) - 1], bs)[0]
            assert len(s.table) == s.blocks_needed


def test_small_trace_invariants_and_completion():
    bs = 16
    steps, prefills, finished = 0, 0, {}
    sched = None
    for st, sched in E.engine_trace(num_requests=24, max_num_batched_tokens=512, max_num_seqs=16,
                                    num_blocks=40, block_size=bs, prompt_range=(5, 120),
                                    output_range=(5, 60)):
        _check_step(st, sched, bs)
        steps += 1
        prefills += st.is_prefill
    assert sched.done() and steps > 50 and prefills >= 2
    assert sched.preemptions > 0, "the small pool must force preemption"
    assert sched.pool.num_free == 40


def test_every_request_gets_exactly_max_tokens():
    """A sequence is scheduled until its last step produces token number
    max_tokens (prefill steps emit a token too, re-prefills included)."""
    reqs = E.make_requests(12, (5, 40), (3, 30))
    counts = {}
    for st, sched in E.engine_trace(num_requests=12, max_num_batched_tokens=256, max_num_seqs=8,
                                    num_blocks=12, block_size=16, prompt_range=(5, 40),
                                    output_range=(3, 30)):
        for sid in st.seq_ids:
            s = next(x for x in list(sched.running) if x.rid == sid)
            counts[sid] = s.generated + 1
    for i, (toks, out_len) in enumerate(reqs):
        assert counts[i] == out_len


def test_prefix_cache_hits_after_preemption_are_consistent():
    """Re-prefill after preemption may hit blocks still holding its K/V; a hit
    always covers whole blocks and the hit block's token ids match."""
    hits = 0
    for st, sched in E.engine_trace(num_requests=20, max_num_batched_tokens=400, max_num_seqs=12,
                                    num_blocks=24, block_size=16, prompt_range=(20, 90),
                                    output_range=(10, 60)):
        if st.is_prefill:
            for sid in st.seq_ids:
                s = next(x for x in sched.running if x.rid == sid)
                assert s.cached % 16 == 0
                for i in range(s.cached_blocks):
                    assert sched.pool.content[s.table[i]] == s.block_tokens(i)
                hits += s.cached_blocks
    assert hits > 0


def test_chained_hash_distinguishes_prefixes():
    """Pages' example: [A, B, C] and [A, B, D] share the hashes of their first
    two blocks and differ on the third."""
    A, B, C, D = [1] * 4, [2] * 4, [3] * 4, [4] * 4
    h = E.chain_hash
    ha = h(A)
    hb = h(B, ha)
    assert h(B, h(A)) == hb and h(C, hb) != h(D, hb) and h(B) != hb


@pytest.mark.slow
def test_full_trace_config5_invariants():
    """256 requests, prompts and outputs U[100, 1024], 768-block pool of 256
    tokens, max_num_batched_tokens 16384, max_num_seqs 512."""
    n = 0
    for st, sched in E.engine_trace():
        if n % 25 == 0:
            _check_step(st, sched, 256)
        n += 1
    assert sched.done() and sched.preemptions > 0
