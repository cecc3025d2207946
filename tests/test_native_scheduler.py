"""The native (C++) block manager and scheduler, through its C ABI, against
the Python replica of the pages' policy (engine_trace.py): step by step the
same sequences are scheduled, with the same cached-prefix lengths, block
tables, attention metadata and preemption counts.  Host only."""
import numpy as np
import pytest
import torch

from paged_kv_cache_125_gb300 import engine_trace as E
from paged_kv_cache_125_gb300 import workloads as W
from paged_kv_cache_125_gb300.scheduler import NativeScheduler


def _same_meta(a, b, is_prefill):
    if is_prefill:
        assert torch.equal(a.cu_seqlens_q, b.cu_seqlens_q) and torch.equal(a.cu_seqlens_k, b.cu_seqlens_k)
        assert (a.max_seqlen_q, a.max_seqlen_k) == (b.max_seqlen_q, b.max_seqlen_k)
        assert (a.block_tables is None) == (b.block_tables is None)
        if a.block_tables is not None:
            assert torch.equal(a.block_tables, b.block_tables)
    else:
        assert torch.equal(a.context_lens, b.context_lens) and a.max_context_len == b.max_context_len
        assert torch.equal(a.block_tables, b.block_tables)
    assert torch.equal(a.positions, b.positions) and torch.equal(a.slot_mapping, b.slot_mapping)


def _replay(requests, num_blocks, block_size, max_num_seqs, max_batched, max_steps=100000):
    py = E.Scheduler(max_num_seqs, max_batched, num_blocks, block_size)
    nat = NativeScheduler(num_blocks, block_size, max_num_seqs, max_batched)
    for i, (toks, out_len) in enumerate(requests):
        py.submit(E.Request(i, toks, out_len, block_size))
        nat.add(i, toks, out_len)
    steps = prefills = 0
    while not py.done():
        assert not nat.is_finished()
        seqs, is_prefill = py.next_batch()
        ids, nat_prefill, meta = nat.step()
        assert ids == [s.rid for s in seqs] and nat_prefill == is_prefill, steps
        if is_prefill:
            ref = W.prefill_metadata([len(s) for s in seqs], [s.cached for s in seqs],
                                     [list(s.table) for s in seqs], block_size)
            prefills += 1
        else:
            ref = W.decode_metadata([len(s) for s in seqs], [list(s.table) for s in seqs],
                                    block_size)
        _same_meta(meta, ref, is_prefill)
        for s in seqs:
            st = nat.seq_state(s.rid)
            assert st["num_cached_tokens"] == s.cached and st["block_table"] == s.table
        assert nat.num_preemptions == py.preemptions
        assert nat.num_free_blocks == py.pool.num_free
        toks = [E.synthetic_token(s.rid, len(s)) for s in seqs]
        py.commit(seqs, toks)
        nat.postprocess(toks)
        steps += 1
        assert steps < max_steps
    assert nat.is_finished()
    return steps, prefills, py.preemptions


def test_small_pool_with_preemption_matches_python_replica():
    reqs = E.make_requests(64, (20, 200), (10, 80))
    steps, prefills, pre = _replay(reqs, num_blocks=64, block_size=16, max_num_seqs=32, max_batched=1024)
    assert pre > 0 and prefills > 1


def test_shared_prefixes_hit_the_cache_like_the_replica():
    g = torch.Generator().manual_seed(9)
    base = torch.randint(0, 1000, (50,), generator=g).tolist()
    reqs = []
    for i in range(12):
        tail = torch.randint(0, 1000, (int(torch.randint(1, 40, (1,), generator=g)),), generator=g).tolist()
        reqs.append((base + tail, 5 + i))
    # a few identical prompts: every full block hits
    reqs += [(list(base[:48]), 3)] * 3
    _replay(reqs, num_blocks=48, block_size=16, max_num_seqs=4, max_batched=256)


@pytest.mark.parametrize("bs", [16, 256])
def test_engine_trace_configuration_matches_python_replica(bs):
    """The engine-trace configuration's request set (256 requests, prompts and
    outputs U[100, 1024]) on its 768-block pool of 256 tokens, and on a
    16-token-block pool of the same byte size."""
    reqs = E.make_requests(256, (100, 1024), (100, 1024))
    nb = 768 * 256 // bs
    steps, prefills, pre = _replay(reqs, num_blocks=nb, block_size=bs, max_num_seqs=512, max_batched=16384)
    if bs == 256:  # the configuration's pool runs out: the replica preempts 80 times
        assert pre == 80
