"""Policy pins for the scheduler / block manager, worked out by hand from the
rules the pages state ("nano-vLLM-1", Scheduler "2. prefill 的 schedule",
"3. decode 的 schedule", "4. 后处理：postprocess()"; BlockManager "3. 核心方法一：
分配 (allocate)", "4. 核心方法二：追加 (may_append)", "5. 核心方法三：回收块
（deallocate）"), not produced by running either scheduler.  Each trace is
replayed by the Python replica (engine_trace.py) and by the native C++
scheduler, and every step must match the hand-worked expectation: which
requests run, prefill or decode, cached prefix, block tables, slot_mapping,
cu_seqlens / context_lens, the free-block queue and the preemption count.

Trace 1 pins the prefill budget (it tests a request's full length but charges
only its uncached tokens) and the FIFO free list.  Trace 2 pins a decode
request evicting itself when nobody is left to evict, and a freed block that
was reused (its old hash no longer hits).  Trace 3 pins eviction of the tail
of the running queue.  Host only."""
import pytest
import torch

from paged_kv_cache_125_gb300 import engine_trace as E
from paged_kv_cache_125_gb300.scheduler import NativeScheduler

# Each step: (is_prefill, request ids, cached tokens per request (prefill only),
#             block tables, slot_mapping, cu_seqlens_q/k (prefill) or context_lens (decode),
#             tokens the step samples, free queue after the step, preemptions after the step)
TRACE1 = dict(
    block_size=4, num_blocks=7, max_num_seqs=4, max_batched=18,
    requests=[([1, 2, 3, 4, 5, 6, 7, 8], 3),        # R0: two full blocks
              ([1, 2, 3, 4, 5, 6, 7, 8, 9], 2),     # R1: R0's blocks + one token
              ([20, 21, 22], 1),                    # R2
              ([1, 2, 3, 4, 5, 6, 7, 8, 30], 1)],   # R3: R0's blocks + one token
    steps=[
        # R0 charges 8; R1 passes the test (8 + 9 <= 18), hits both of R0's blocks and is
        # charged 1; R2 passes (9 + 3 <= 18; it would not if R1 had been charged 9); R3 fails
        # the test on its full length (12 + 9 > 18) although its uncached part would fit.
        (True, [0, 1, 2], [0, 8, 0], [[0, 1], [0, 1, 2], [3]],
         [0, 1, 2, 3, 4, 5, 6, 7, 8, 12, 13, 14], ([0, 8, 9, 12], [0, 8, 17, 20]),
         [100, 101, 102], [4, 5, 6, 3], 0),
        # R2 finished and its block 3 went to the back of the queue: R3's fresh block is 4
        # (the front), not 3.
        (True, [3], [8], [[0, 1, 4]], [16], ([0, 1], [0, 9]), [113], [5, 6, 3, 4], 0),
        # R0's 9th token opens a block (front: 5); R1's 10th does not.
        (False, [0, 1], None, [[0, 1, 5], [0, 1, 2]], [20, 9], [9, 10], [120, 121], [6, 3, 4, 2], 0),
        (False, [0], None, [[0, 1, 5]], [21], [10], [130], [6, 3, 4, 2, 5, 1, 0], 0),
    ])

TRACE2 = dict(
    block_size=2, num_blocks=3, max_num_seqs=4, max_batched=100,
    requests=[([1, 2, 3], 3), ([4, 5], 3)],
    steps=[
        (True, [0, 1], [0, 0], [[0, 1], [2]], [0, 1, 2, 4, 5], ([0, 3, 5], [0, 3, 5]), [7, 8], [], 0),
        # B's 3rd token needs a block, none is free and the running queue is empty (A was
        # taken first): B evicts itself; its block 2 returns to the queue.
        (False, [0], None, [[0, 1]], [3], [4], [9], [2], 1),
        # B (3 tokens, 2 blocks) does not fit in 1 free block: no prefill; A takes block 2.
        (False, [0], None, [[0, 1, 2]], [4], [5], [11], [2, 1, 0], 1),
        # B's first block [4, 5] was indexed at block 2, which A reused: a miss.
        (True, [1], [0], [[2, 1]], [4, 5, 2], ([0, 3], [0, 3]), [12], [0], 1),
        (False, [1], None, [[2, 1]], [3], [4], [13], [0, 1, 2], 1),
    ])

TRACE3 = dict(
    block_size=2, num_blocks=2, max_num_seqs=4, max_batched=100,
    requests=[([1], 3), ([2], 3)],
    steps=[
        (True, [0, 1], [0, 0], [[0], [1]], [0, 2], ([0, 1, 2], [0, 1, 2]), [5, 6], [], 0),
        (False, [0, 1], None, [[0], [1]], [1, 3], [2, 2], [7, 8], [], 0),
        # A's 3rd token needs a block: the tail of the running queue (B) is evicted.
        (False, [0], None, [[0, 1]], [2], [3], [9], [1, 0], 1),
        # B's re-prefill samples its 3rd token (two came before the eviction): it finishes and
        # releases its blocks last block first.
        (True, [1], [0], [[1, 0]], [2, 3, 0], ([0, 3], [0, 3]), [10], [0, 1], 1),
    ])


def _tables(rows):
    return [list(r) for r in rows]


def _check_meta(meta, exp, is_prefill):
    assert meta.slot_mapping.tolist() == exp[4]
    if is_prefill:
        assert (meta.cu_seqlens_q.tolist(), meta.cu_seqlens_k.tolist()) == tuple(exp[5])
        if exp[2] is not None and any(exp[2]):
            width = max(len(t) for t in exp[3])
            want = [t + [-1] * (width - len(t)) for t in exp[3]]
            assert meta.block_tables.tolist() == want
        else:
            assert meta.block_tables is None
    else:
        assert meta.context_lens.tolist() == exp[5]
        width = max(len(t) for t in exp[3])
        assert meta.block_tables.tolist() == [t + [-1] * (width - len(t)) for t in exp[3]]


@pytest.mark.parametrize("trace", [TRACE1, TRACE2, TRACE3], ids=["budget_fifo", "self_evict", "tail_evict"])
def test_python_replica_follows_the_hand_worked_trace(trace):
    bs = trace["block_size"]
    sch = E.Scheduler(trace["max_num_seqs"], trace["max_batched"], trace["num_blocks"], bs)
    for i, (toks, n) in enumerate(trace["requests"]):
        sch.submit(E.Request(i, toks, n, bs))
    for k, exp in enumerate(trace["steps"]):
        batch, pre = sch.next_batch()
        assert (pre, [r.rid for r in batch]) == (exp[0], exp[1]), f"step {k}"
        if pre:
            assert [r.cached for r in batch] == exp[2], f"step {k}"
        assert _tables(r.table for r in batch) == exp[3], f"step {k}"
        meta, _ = E.step_metadata(batch, pre, bs)
        _check_meta(meta, exp, pre)
        sch.commit(batch, exp[6])
        assert list(sch.pool.free_queue) == exp[7], f"step {k}"
        assert sch.preemptions == exp[8], f"step {k}"
    assert sch.done()


@pytest.mark.parametrize("trace", [TRACE1, TRACE2, TRACE3], ids=["budget_fifo", "self_evict", "tail_evict"])
def test_native_scheduler_follows_the_hand_worked_trace(trace):
    bs = trace["block_size"]
    nat = NativeScheduler(trace["num_blocks"], bs, trace["max_num_seqs"], trace["max_batched"])
    for i, (toks, n) in enumerate(trace["requests"]):
        nat.add(i, toks, n)
    for k, exp in enumerate(trace["steps"]):
        ids, pre, meta = nat.step()
        assert (pre, ids) == (exp[0], exp[1]), f"step {k}"
        states = [nat.seq_state(i) for i in ids]
        if pre:
            assert [s["num_cached_tokens"] for s in states] == exp[2], f"step {k}"
        assert [list(s["block_table"]) for s in states] == exp[3], f"step {k}"
        _check_meta(meta, exp, pre)
        nat.postprocess(exp[6])
        assert nat.num_free_blocks == len(exp[7]), f"step {k}"
        assert nat.num_preemptions == exp[8], f"step {k}"
    assert nat.is_finished()
