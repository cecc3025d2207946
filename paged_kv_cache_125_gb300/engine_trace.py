"""Engine-step trace of a nano-vLLM-style scheduler, for replaying the hot path.

Host-side input generation: a replica of the pages' scheduling policy
("nano-vLLM-1", Scheduler sections "1. 队列与状态机", "2. prefill 的 schedule",
"3. decode 的 schedule", "4. 后处理：postprocess()"; BlockManager sections
"1. Block", "2. BlockManager 初始化与链式哈希", "3. 核心方法一：分配 (allocate)",
"4. 核心方法二：追加 (may_append)", "5. 核心方法三：回收块（deallocate）",
"6. 辅助查询方法"; the Sequence section) that turns a seeded set of requests
into the sequence of engine steps, each with the metadata the ModelRunner
builds for the attention kernels (``workloads.prefill_metadata`` /
``workloads.decode_metadata``).  No attention arithmetic lives here.

Policy, as the pages state it:
* prefill first: FCFS from the head of ``waiting``; stop at the first
  sequence whose full length would exceed max_num_batched_tokens or that
  can_allocate rejects; the budget is charged len - num_cached_tokens; a step
  that schedules any prefill is a prefill-only step;
* otherwise decode: pop from the head of ``running``; while the sequence cannot
  append, preempt the tail of ``running`` (or the sequence itself when it is
  alone); may_append; the scheduled sequences go back to the head in order;
* preemption frees the sequence's blocks and puts it at the head of
  ``waiting`` (it is prefilled again later);
* postprocess appends the step's token; a sequence finishes at max_tokens
  (ignore_eos is set: synthetic tokens carry no EOS);
* blocks: FIFO free list; a full block's chained hash (prefix hash, 8 bytes
  little-endian, then the token ids) is registered for prefix caching; a hit
  is confirmed by comparing token ids; freed blocks keep their hash, so a
  re-prefill after preemption can hit them.  xxhash is not available here, so
  the 64-bit hash is blake2b with an 8-byte digest (any 64-bit hash works
  because hits compare the token ids).
"""
from __future__ import annotations

import hashlib
from collections import deque
from dataclasses import dataclass
from enum import Enum, auto

import numpy as np
import torch

from . import workloads as W


class Status(Enum):
    WAITING = auto()
    RUNNING = auto()
    FINISHED = auto()


class Sequence:
    def __init__(self, seq_id: int, token_ids: list[int], max_tokens: int, block_size: int):
        self.seq_id = seq_id
        self.block_size = block_size
        self.status = Status.WAITING
        self.token_ids = list(token_ids)
        self.last_token = token_ids[-1]
        self.num_tokens = len(token_ids)
        self.num_prompt_tokens = len(token_ids)
        self.num_cached_tokens = 0
        self.block_table: list[int] = []
        self.max_tokens = max_tokens
        self.ignore_eos = True

    def __len__(self):
        return self.num_tokens

    @property
    def num_completion_tokens(self):
        return self.num_tokens - self.num_prompt_tokens

    @property
    def num_cached_blocks(self):
        return self.num_cached_tokens // self.block_size

    @property
    def num_blocks(self):
        return (self.num_tokens + self.block_size - 1) // self.block_size

    @property
    def last_block_num_tokens(self):
        return self.num_tokens - (self.num_blocks - 1) * self.block_size

    def block(self, i):
        assert 0 <= i < self.num_blocks
        return self.token_ids[i * self.block_size:(i + 1) * self.block_size]

    def append_token(self, token_id: int):
        self.token_ids.append(token_id)
        self.last_token = token_id
        self.num_tokens += 1


class Block:
    def __init__(self, block_id: int):
        self.block_id = block_id
        self.ref_count = 0
        self.hash = -1
        self.token_ids: list[int] = []

    def update(self, h: int, token_ids: list[int]):
        self.hash = h
        self.token_ids = token_ids

    def reset(self):
        self.ref_count = 1
        self.hash = -1
        self.token_ids = []


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        self.block_size = block_size
        self.blocks = [Block(i) for i in range(num_blocks)]
        self.hash_to_block_id: dict[int, int] = {}
        self.free_block_ids: deque[int] = deque(range(num_blocks))
        self.used_block_ids: set[int] = set()

    @staticmethod
    def compute_hash(token_ids: list[int], prefix: int = -1) -> int:
        h = hashlib.blake2b(digest_size=8)
        if prefix != -1:
            h.update(prefix.to_bytes(8, "little"))
        h.update(np.asarray(token_ids, dtype=np.int64).tobytes())
        return int.from_bytes(h.digest(), "little")

    def _allocate_block(self, block_id: int) -> Block:
        block = self.blocks[block_id]
        assert block.ref_count == 0
        block.reset()
        self.free_block_ids.remove(block_id)
        self.used_block_ids.add(block_id)
        return block

    def _deallocate_block(self, block_id: int):
        assert self.blocks[block_id].ref_count == 0
        self.used_block_ids.remove(block_id)
        self.free_block_ids.append(block_id)

    def can_allocate(self, seq: Sequence) -> bool:
        return len(self.free_block_ids) >= seq.num_blocks

    def allocate(self, seq: Sequence):
        assert not seq.block_table
        h = -1
        cache_miss = False
        for i in range(seq.num_blocks):
            token_ids = seq.block(i)
            h = self.compute_hash(token_ids, h) if len(token_ids) == self.block_size else -1
            block_id = self.hash_to_block_id.get(h, -1)
            if block_id == -1 or self.blocks[block_id].token_ids != token_ids:
                cache_miss = True
            if cache_miss:
                block = self._allocate_block(self.free_block_ids[0])
            else:
                seq.num_cached_tokens += self.block_size
                if block_id in self.used_block_ids:
                    block = self.blocks[block_id]
                    block.ref_count += 1
                else:
                    block = self._allocate_block(block_id)
            if h != -1:
                block.update(h, token_ids)
                self.hash_to_block_id[h] = block.block_id
            seq.block_table.append(block.block_id)

    def deallocate(self, seq: Sequence):
        for block_id in reversed(seq.block_table):
            block = self.blocks[block_id]
            block.ref_count -= 1
            if block.ref_count == 0:
                self._deallocate_block(block_id)
        seq.num_cached_tokens = 0
        seq.block_table.clear()

    def can_append(self, seq: Sequence) -> bool:
        return len(self.free_block_ids) >= (len(seq) % self.block_size == 1)

    def may_append(self, seq: Sequence):
        table = seq.block_table
        last = self.blocks[table[-1]]
        if len(seq) % self.block_size == 1:
            assert last.hash != -1
            block_id = self.free_block_ids[0]
            self._allocate_block(block_id)
            table.append(block_id)
        elif len(seq) % self.block_size == 0:
            assert last.hash == -1
            token_ids = seq.block(seq.num_blocks - 1)
            prefix = self.blocks[table[-2]].hash if len(table) > 1 else -1
            h = self.compute_hash(token_ids, prefix)
            last.update(h, token_ids)
            self.hash_to_block_id[h] = last.block_id
        else:
            assert last.hash == -1


class Scheduler:
    def __init__(self, max_num_seqs: int, max_num_batched_tokens: int, num_blocks: int,
                 block_size: int):
        self.max_num_seqs = max_num_seqs
        self.max_num_batched_tokens = max_num_batched_tokens
        self.block_manager = BlockManager(num_blocks, block_size)
        self.waiting: deque[Sequence] = deque()
        self.running: deque[Sequence] = deque()
        self.num_preemptions = 0

    def is_finished(self):
        return not self.waiting and not self.running

    def add(self, seq: Sequence):
        self.waiting.append(seq)

    def preempt(self, seq: Sequence):
        seq.status = Status.WAITING
        self.block_manager.deallocate(seq)
        self.waiting.appendleft(seq)
        self.num_preemptions += 1

    def schedule(self) -> tuple[list[Sequence], bool]:
        scheduled: list[Sequence] = []
        num_seqs = 0
        num_batched_tokens = 0
        while self.waiting and num_seqs < self.max_num_seqs:
            seq = self.waiting[0]
            if (num_batched_tokens + len(seq) > self.max_num_batched_tokens
                    or not self.block_manager.can_allocate(seq)):
                break
            num_seqs += 1
            self.block_manager.allocate(seq)
            num_batched_tokens += len(seq) - seq.num_cached_tokens
            seq.status = Status.RUNNING
            self.waiting.popleft()
            self.running.append(seq)
            scheduled.append(seq)
        if scheduled:
            return scheduled, True
        while self.running and num_seqs < self.max_num_seqs:
            seq = self.running.popleft()
            while not self.block_manager.can_append(seq):
                if self.running:
                    self.preempt(self.running.pop())
                else:
                    self.preempt(seq)
                    break
            else:
                num_seqs += 1
                self.block_manager.may_append(seq)
                scheduled.append(seq)
        assert scheduled, "nothing schedulable: the pool cannot hold a single sequence"
        self.running.extendleft(reversed(scheduled))
        return scheduled, False

    def postprocess(self, seqs: list[Sequence], token_ids: list[int]):
        for seq, tok in zip(seqs, token_ids):
            seq.append_token(tok)
            if seq.num_completion_tokens == seq.max_tokens:
                seq.status = Status.FINISHED
                self.block_manager.deallocate(seq)
                self.running.remove(seq)


# ---------------------------------------------------------------------------

@dataclass
class TraceStep:
    index: int
    is_prefill: bool
    seq_ids: list[int]
    meta: object            # workloads.PrefillMeta or workloads.DecodeMeta
    num_new_tokens: int     # rows stored (and queried) this step
    preempted_so_far: int


def synthetic_token(seq_id: int, position: int, vocab: int = 151936) -> int:
    """Deterministic stand-in for the sampled token at (sequence, position)."""
    h = hashlib.blake2b(f"{seq_id}:{position}".encode(), digest_size=4).digest()
    return int.from_bytes(h, "little") % vocab


def make_requests(num_requests=256, prompt_range=(100, 1024), output_range=(100, 1024),
                  vocab=151936):
    g = W.generator(W.SEED_LENGTHS)
    prompts = torch.randint(prompt_range[0], prompt_range[1] + 1, (num_requests,), generator=g).tolist()
    outputs = torch.randint(output_range[0], output_range[1] + 1, (num_requests,), generator=g).tolist()
    gt = W.generator(W.SEED_TOKENS)
    reqs = []
    for i, (p, o) in enumerate(zip(prompts, outputs)):
        toks = torch.randint(0, vocab, (p,), generator=gt).tolist()
        reqs.append((toks, o))
    return reqs


def engine_trace(num_requests=256, max_num_batched_tokens=16384, max_num_seqs=512, num_blocks=768,
                 block_size=256, prompt_range=(100, 1024), output_range=(100, 1024), max_steps=None):
    """Yields the engine's steps for the seeded request set, with the attention
    metadata of each step (the pages' prepare_prefill / prepare_decode)."""
    sched = Scheduler(max_num_seqs, max_num_batched_tokens, num_blocks, block_size)
    for i, (toks, out_len) in enumerate(make_requests(num_requests, prompt_range, output_range)):
        sched.add(Sequence(i, toks, out_len, block_size))
    step = 0
    while not sched.is_finished():
        if max_steps is not None and step >= max_steps:
            return
        seqs, is_prefill = sched.schedule()
        if is_prefill:
            meta = W.prefill_metadata([len(s) for s in seqs], [s.num_cached_tokens for s in seqs],
                                      [list(s.block_table) for s in seqs], block_size)
            n_new = int(meta.cu_seqlens_q[-1])
        else:
            meta = W.decode_metadata([len(s) for s in seqs], [list(s.block_table) for s in seqs],
                                     block_size)
            n_new = len(seqs)
        yield TraceStep(step, is_prefill, [s.seq_id for s in seqs], meta, n_new, sched.num_preemptions), sched
        sched.postprocess(seqs, [synthetic_token(s.seq_id, len(s)) for s in seqs])
        step += 1
