"""Engine-step trace of a nano-vLLM-style scheduler, for replaying the hot path.

Host-side input generation.  It turns a seeded set of requests into the
sequence of engine steps the pages' scheduling policy produces, each with the
metadata the ModelRunner builds for the attention kernels
(``workloads.prefill_metadata`` / ``workloads.decode_metadata``).  No attention
arithmetic lives here.

The policy, as "nano-vLLM-1" states it (Scheduler: "1. 队列与状态机",
"2. prefill 的 schedule", "3. decode 的 schedule", "4. 后处理：postprocess()";
BlockManager: "1. Block" .. "6. 辅助查询方法"; Sequence), restated here as
rules and implemented in a structure of this module's own:

Pool of physical blocks (``KVPool``)
  P1  Free blocks form a FIFO queue: a fresh block is taken from the front,
      a released block goes to the back.
  P2  A block is in use while its reference count is positive.
  P3  A full block carries a chain hash: hash(previous full block's hash as 8
      little-endian bytes, then the block's token ids); the first block has no
      previous hash.  The pool indexes full blocks by that hash.  A lookup is a
      hit only if the indexed block still holds the same token ids.
  P4  Placing a prompt: walking its blocks in order, every block up to the
      first miss is shared (reference + 1 if in use; taken back out of the free
      queue, wherever it sits, if it was free); from the first miss on (a
      partial last block always misses) every block is a fresh one.  Each hit
      adds a whole block to the request's cached tokens.  Every full block is
      (re)registered under its hash.  A fresh block forgets what it held.
  P5  Releasing a request drops one reference per block, last block first;
      blocks that reach zero return to the free queue and keep their hash and
      token ids, so a later prompt (a re-prefill after preemption) can hit them.
  P6  A decode step's new token needs a fresh block when it is the first token
      of a block (length % block_size == 1); when it fills a block
      (length % block_size == 0) that block's hash is registered.
Scheduler (``Scheduler``)
  S1  Prefill first.  From the head of the waiting queue, in order, admit a
      request if (tokens charged so far + its FULL length) stays within
      max_num_batched_tokens and the pool has at least as many free blocks as
      the request has blocks (cache hits are not discounted); charge it only
      its uncached tokens.  The first request that fails either test ends the
      batch, as does max_num_seqs.  A step that admits anything is a
      prefill-only step.
  S2  Otherwise decode: take requests from the head of the running queue.
      While a request's next token needs a block and none is free, evict the
      tail of the running queue; with nobody left to evict, evict the request
      itself (it is not scheduled).  The scheduled requests go back to the
      head of the running queue in their order.
  S3  Eviction (preemption) releases the request's blocks and puts it at the
      head of the waiting queue; it is prefilled again later.
  S4  After a step every scheduled request gets one token; a request that
      reaches its max_tokens finishes and releases its blocks (ignore_eos:
      synthetic tokens carry no EOS).
xxhash is not available here, so the 64-bit hash is blake2b with an 8-byte
digest; any 64-bit hash gives the same schedule because hits compare token ids.
"""
from __future__ import annotations

import hashlib
from collections import deque
from dataclasses import dataclass, field

import numpy as np
import torch

from . import workloads as W

WAITING, RUNNING, FINISHED = "waiting", "running", "finished"


def chain_hash(tokens, prev: int | None = None) -> int:
    """Rule P3: 64-bit hash of (previous block's hash, this block's token ids)."""
    h = hashlib.blake2b(digest_size=8)
    if prev is not None:
        h.update(prev.to_bytes(8, "little"))
    h.update(np.asarray(tokens, dtype=np.int64).tobytes())
    return int.from_bytes(h.digest(), "little")


@dataclass
class Request:
    """One sequence: its prompt and generated token ids, and its place in the pool."""
    rid: int
    tokens: list[int]
    max_tokens: int
    block_size: int
    cached: int = 0                                    # tokens served from the prefix cache
    table: list[int] = field(default_factory=list)     # physical block ids, logical order
    state: str = WAITING
    prompt_len: int = 0

    def __post_init__(self):
        self.tokens = list(self.tokens)
        self.prompt_len = len(self.tokens)

    def __len__(self) -> int:
        return len(self.tokens)

    @property
    def generated(self) -> int:
        return len(self.tokens) - self.prompt_len

    @property
    def blocks_needed(self) -> int:
        return W.num_blocks_for(len(self.tokens), self.block_size)

    @property
    def cached_blocks(self) -> int:
        return self.cached // self.block_size

    def block_tokens(self, i: int) -> list[int]:
        bs = self.block_size
        return self.tokens[i * bs:(i + 1) * bs]


class KVPool:
    """Physical blocks of the KV cache: rules P1-P6."""

    def __init__(self, num_blocks: int, block_size: int):
        self.block_size = block_size
        self.refs = [0] * num_blocks
        self.key: list[int | None] = [None] * num_blocks        # registered chain hash
        self.content: list[list[int] | None] = [None] * num_blocks  # token ids behind it
        self.index: dict[int, int] = {}                         # chain hash -> block id
        self.free_queue: deque[int] = deque(range(num_blocks))  # P1: front = next fresh block

    @property
    def num_blocks(self) -> int:
        return len(self.refs)

    @property
    def num_free(self) -> int:
        return len(self.free_queue)

    def in_use(self) -> set[int]:
        return {b for b, r in enumerate(self.refs) if r > 0}

    def _claim(self, bid: int) -> int:
        """A free block becomes a fresh, single-owner block (P4: it forgets its content)."""
        assert self.refs[bid] == 0, f"block {bid} is in use"
        self.free_queue.remove(bid)
        self.refs[bid] = 1
        self.key[bid] = None
        self.content[bid] = None
        return bid

    def _register(self, bid: int, h: int, tokens: list[int]):
        self.key[bid] = h
        self.content[bid] = list(tokens)
        self.index[h] = bid

    def _lookup(self, h: int | None, tokens: list[int]) -> int | None:
        if h is None:
            return None
        bid = self.index.get(h)
        return bid if bid is not None and self.content[bid] == tokens else None

    def fits_prompt(self, req: Request) -> bool:
        return self.num_free >= req.blocks_needed

    def place_prompt(self, req: Request):
        """P4."""
        assert not req.table
        prev, missed = None, False
        for i in range(req.blocks_needed):
            toks = req.block_tokens(i)
            h = chain_hash(toks, prev) if len(toks) == self.block_size else None
            hit = None if missed else self._lookup(h, toks)
            if hit is None:
                missed = True
                bid = self._claim(self.free_queue[0])
            else:
                req.cached += self.block_size
                bid = hit
                if self.refs[bid] > 0:
                    self.refs[bid] += 1
                else:
                    self._claim(bid)
            if h is not None:
                self._register(bid, h, toks)
            req.table.append(bid)
            prev = h

    def release(self, req: Request):
        """P5."""
        for bid in reversed(req.table):
            self.refs[bid] -= 1
            if self.refs[bid] == 0:
                self.free_queue.append(bid)
        req.table = []
        req.cached = 0

    def fits_next_token(self, req: Request) -> bool:
        return self.num_free >= (1 if len(req) % self.block_size == 1 else 0)

    def on_next_token(self, req: Request):
        """P6, for the token at position len(req) - 1."""
        phase = len(req) % self.block_size
        if phase == 1:
            req.table.append(self._claim(self.free_queue[0]))
        elif phase == 0:
            last = req.blocks_needed - 1
            prev = self.key[req.table[last - 1]] if last > 0 else None
            self._register(req.table[last], chain_hash(req.block_tokens(last), prev),
                           req.block_tokens(last))


class Scheduler:
    """Rules S1-S4 over a KVPool."""

    def __init__(self, max_num_seqs: int, max_num_batched_tokens: int, num_blocks: int,
                 block_size: int):
        self.max_num_seqs = max_num_seqs
        self.max_num_batched_tokens = max_num_batched_tokens
        self.pool = KVPool(num_blocks, block_size)
        self.waiting: deque[Request] = deque()
        self.running: deque[Request] = deque()
        self.preemptions = 0

    def submit(self, req: Request):
        self.waiting.append(req)

    def done(self) -> bool:
        return not self.waiting and not self.running

    def next_batch(self) -> tuple[list[Request], bool]:
        batch = self._prefill_batch()
        if batch:
            return batch, True
        return self._decode_batch(), False

    def _prefill_batch(self) -> list[Request]:
        """S1."""
        batch: list[Request] = []
        charged = 0
        while self.waiting and len(batch) < self.max_num_seqs:
            req = self.waiting[0]
            if charged + len(req) > self.max_num_batched_tokens or not self.pool.fits_prompt(req):
                break
            self.pool.place_prompt(req)
            charged += len(req) - req.cached
            self.waiting.popleft()
            req.state = RUNNING
            self.running.append(req)
            batch.append(req)
        return batch

    def _decode_batch(self) -> list[Request]:
        """S2."""
        batch: list[Request] = []
        while self.running and len(batch) < self.max_num_seqs:
            req = self.running.popleft()
            if self._make_room(req):
                self.pool.on_next_token(req)
                batch.append(req)
        assert batch, "nothing schedulable: the pool cannot hold a single sequence"
        self.running = deque(batch + list(self.running))
        return batch

    def _make_room(self, req: Request) -> bool:
        while not self.pool.fits_next_token(req):
            if not self.running:
                self._evict(req)
                return False
            self._evict(self.running.pop())
        return True

    def _evict(self, req: Request):
        """S3."""
        req.state = WAITING
        self.pool.release(req)
        self.waiting.appendleft(req)
        self.preemptions += 1

    def commit(self, batch: list[Request], tokens: list[int]):
        """S4."""
        for req, tok in zip(batch, tokens):
            req.tokens.append(tok)
            if req.generated == req.max_tokens:
                req.state = FINISHED
                self.pool.release(req)
                self.running.remove(req)


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
    for p, o in zip(prompts, outputs):
        toks = torch.randint(0, vocab, (p,), generator=gt).tolist()
        reqs.append((toks, o))
    return reqs


def step_metadata(batch: list[Request], is_prefill: bool, block_size: int):
    """The ModelRunner's metadata for one scheduled batch -> (meta, new rows)."""
    lens, tables = [len(r) for r in batch], [list(r.table) for r in batch]
    if is_prefill:
        meta = W.prefill_metadata(lens, [r.cached for r in batch], tables, block_size)
        return meta, int(meta.cu_seqlens_q[-1])
    return W.decode_metadata(lens, tables, block_size), len(batch)


def engine_trace(num_requests=256, max_num_batched_tokens=16384, max_num_seqs=512, num_blocks=768,
                 block_size=256, prompt_range=(100, 1024), output_range=(100, 1024), max_steps=None):
    """Yields (TraceStep, scheduler) for every engine step of the seeded request
    set, with the attention metadata of each step."""
    sched = Scheduler(max_num_seqs, max_num_batched_tokens, num_blocks, block_size)
    for i, (toks, out_len) in enumerate(make_requests(num_requests, prompt_range, output_range)):
        sched.submit(Request(i, toks, out_len, block_size))
    step = 0
    while not sched.done():
        if max_steps is not None and step >= max_steps:
            return
        batch, is_prefill = sched.next_batch()
        meta, n_new = step_metadata(batch, is_prefill, block_size)
        yield TraceStep(step, is_prefill, [r.rid for r in batch], meta, n_new, sched.preemptions), sched
        sched.commit(batch, [synthetic_token(r.rid, len(r)) for r in batch])
        step += 1
