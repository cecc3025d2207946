"""Seeded synthetic workloads for the paged KV-cache attention path.

Input generation only.  This module draws the seeded inputs (queries, the new
K/V rows of a step, cached history, sequence lengths, block permutations) and
builds each step's metadata the way the engine's ModelRunner builds it on the
host.  It holds none of the attention arithmetic: the CUDA library's tests and
benchmark, and the CPU oracle, all consume what it produces.

Metadata follows the pages' ModelRunner ("nano-vLLM-1", sections
"4. prefill 输入打包" and "5. deocde 输入打包"; "Nano vLLM 解读（5）：解析
ModelRunner", prepare_prefill / prepare_decode):

* prefill: q covers only the uncached suffix of every sequence
  (q_len = len - num_cached_tokens), k covers the whole prompt (k_len = len);
  cu_seqlens_q / cu_seqlens_k are their prefix sums; slot_mapping lists, block
  by block from the first uncached block, the linear slots block_id * bs + offset
  (the last block only up to last_block_num_tokens); block_tables (right-padded
  with -1) are built only when some prefix was cached (cu_k[-1] > cu_q[-1]);
* decode: one token per sequence at position len - 1, context_lens = len,
  slot = block_table[-1] * bs + last_block_num_tokens - 1, block_tables always.

Seeds: values 0, lengths 1, block permutations 2, token ids 3.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16 = torch.bfloat16
SEED_VALUES, SEED_LENGTHS, SEED_BLOCKS, SEED_TOKENS = 0, 1, 2, 3


def generator(seed: int, device: str | torch.device = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """N(0,1) values drawn in fp32 and rounded to bf16."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(BF16)


# ---------------------------------------------------------------------------
# Sequence bookkeeping of the pages' Sequence class (block_size hard-wired per
# call here instead of the class constant).
# ---------------------------------------------------------------------------

def num_blocks_for(num_tokens: int, block_size: int) -> int:
    return (num_tokens + block_size - 1) // block_size


def last_block_num_tokens(num_tokens: int, block_size: int) -> int:
    return num_tokens - (num_blocks_for(num_tokens, block_size) - 1) * block_size


def prepare_block_tables(tables: list[list[int]]) -> torch.Tensor:
    """Right-pad every block table with -1 to the longest one -> int32 [B, max]."""
    width = max(1, max(len(t) for t in tables))
    return torch.tensor([list(t) + [-1] * (width - len(t)) for t in tables], dtype=torch.int32)


@dataclass
class PrefillMeta:
    cu_seqlens_q: torch.Tensor
    cu_seqlens_k: torch.Tensor
    max_seqlen_q: int
    max_seqlen_k: int
    positions: torch.Tensor
    slot_mapping: torch.Tensor
    block_tables: torch.Tensor | None


def prefill_metadata(seq_lens: list[int], num_cached_tokens: list[int],
                     tables: list[list[int]], block_size: int) -> PrefillMeta:
    cu_q, cu_k, positions, slots = [0], [0], [], []
    max_q = max_k = 0
    for seqlen, cached, bt in zip(seq_lens, num_cached_tokens, tables):
        positions.extend(range(cached, seqlen))
        q_len = seqlen - cached
        cu_q.append(cu_q[-1] + q_len)
        cu_k.append(cu_k[-1] + seqlen)
        max_q, max_k = max(max_q, q_len), max(max_k, seqlen)
        if not bt:
            continue
        nblk = num_blocks_for(seqlen, block_size)
        for i in range(cached // block_size, nblk):
            start = bt[i] * block_size
            end = start + (block_size if i != nblk - 1 else last_block_num_tokens(seqlen, block_size))
            slots.extend(range(start, end))
    block_tables = prepare_block_tables(tables) if cu_k[-1] > cu_q[-1] else None
    return PrefillMeta(torch.tensor(cu_q, dtype=torch.int32), torch.tensor(cu_k, dtype=torch.int32),
                       max_q, max_k, torch.tensor(positions, dtype=torch.int64),
                       torch.tensor(slots, dtype=torch.int32), block_tables)


@dataclass
class DecodeMeta:
    positions: torch.Tensor
    context_lens: torch.Tensor
    slot_mapping: torch.Tensor
    block_tables: torch.Tensor
    max_context_len: int


def decode_metadata(seq_lens: list[int], tables: list[list[int]], block_size: int) -> DecodeMeta:
    positions, ctx, slots = [], [], []
    for seqlen, bt in zip(seq_lens, tables):
        positions.append(seqlen - 1)
        ctx.append(seqlen)
        slots.append(bt[-1] * block_size + last_block_num_tokens(seqlen, block_size) - 1)
    return DecodeMeta(torch.tensor(positions, dtype=torch.int64), torch.tensor(ctx, dtype=torch.int32),
                      torch.tensor(slots, dtype=torch.int32), prepare_block_tables(tables),
                      max(ctx) if ctx else 0)


def slots_of_positions(table: list[int], positions, block_size: int) -> list[int]:
    """Linear slot of each logical position through one block table."""
    return [table[p // block_size] * block_size + p % block_size for p in positions]


# ---------------------------------------------------------------------------
# Calls and workloads
# ---------------------------------------------------------------------------

@dataclass
class StoreCall:
    k: torch.Tensor              # [N, Hkv, d] bf16
    v: torch.Tensor              # [N, Hkv, d] bf16
    slot_mapping: torch.Tensor   # [N] int32, -1 = skip


@dataclass
class PrefillCall:
    q: torch.Tensor              # [sum q, Hq, d] bf16
    k: torch.Tensor              # [sum q, Hkv, d] new rows (also the packed keys without a prefix hit)
    v: torch.Tensor
    meta: PrefillMeta


@dataclass
class DecodeCall:
    q: torch.Tensor              # [B, Hq, d] bf16
    meta: DecodeMeta


@dataclass
class Step:
    store: StoreCall
    attn: PrefillCall | DecodeCall

    @property
    def is_prefill(self) -> bool:
        return isinstance(self.attn, PrefillCall)


@dataclass
class Workload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    steps: list[Step]
    setup: list[StoreCall] = field(default_factory=list)
    # history placed straight into the pool before ``setup`` (decode configs):
    history_slots: torch.Tensor | None = None   # int64 [T]
    history_k: torch.Tensor | None = None       # [T, Hkv, d] bf16
    history_v: torch.Tensor | None = None
    description: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def cache_shape(self):
        return (self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim)

    def new_cache(self, device="cpu", poison: bool = True):
        """Empty K and V pools [NB, bs, Hkv, d]; poisoned with bf16 NaN so that a
        read of any slot never written shows up as NaN downstream."""
        fill = float("nan") if poison else 0.0
        kc = torch.full(self.cache_shape(), fill, dtype=BF16, device=device)
        vc = torch.full(self.cache_shape(), fill, dtype=BF16, device=device)
        return kc, vc

    def place_history(self, k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
        """Copy the pre-existing history rows into their slots (plain tensor
        indexing; this is set-up, not the store kernel)."""
        if self.history_slots is None:
            return
        dev = k_cache.device
        idx = self.history_slots.to(dev)
        hk, hv = self.num_kv_heads, self.head_dim
        k_cache.view(-1, hk, hv).index_copy_(0, idx, self.history_k.to(dev))
        v_cache.view(-1, hk, hv).index_copy_(0, idx, self.history_v.to(dev))


def _assign_blocks(perm: list[int], blocks_needed: list[int]) -> list[list[int]]:
    tables, at = [], 0
    for n in blocks_needed:
        tables.append(perm[at:at + n])
        at += n
    if at > len(perm):
        raise ValueError("block pool too small for the requested sequences")
    return tables


def prefill_workload(name: str, seq_lens: list[int], cached_blocks: list[int], num_heads: int,
                     num_kv_heads: int, head_dim: int, block_size: int, num_blocks: int,
                     extra_decode_steps: int = 0, description: str = "") -> Workload:
    """Prefill of ``seq_lens`` with the first ``cached_blocks[i]`` full blocks of
    sequence i already in the cache (written by a set-up store), optionally
    followed by decode steps on every sequence.  Block tables are consecutive
    slices of one seeded permutation of the pool."""
    gv = generator(SEED_VALUES)
    perm = torch.randperm(num_blocks, generator=generator(SEED_BLOCKS)).tolist()
    final_lens = [L + extra_decode_steps for L in seq_lens]
    tables_full = _assign_blocks(perm, [num_blocks_for(L, block_size) for L in final_lens])
    cached = [c * block_size for c in cached_blocks]
    for L, c in zip(seq_lens, cached):
        if c > L:
            raise ValueError("cached prefix longer than the prompt")

    setup = []
    pre_slots = [s for bt, c in zip(tables_full, cached) for s in slots_of_positions(bt, range(c), block_size)]
    if pre_slots:
        n = len(pre_slots)
        setup.append(StoreCall(randn_bf16((n, num_kv_heads, head_dim), gv),
                               randn_bf16((n, num_kv_heads, head_dim), gv),
                               torch.tensor(pre_slots, dtype=torch.int32)))

    tables_now = [bt[:num_blocks_for(L, block_size)] for bt, L in zip(tables_full, seq_lens)]
    meta = prefill_metadata(seq_lens, cached, tables_now, block_size)
    tq = int(meta.cu_seqlens_q[-1])
    q = randn_bf16((tq, num_heads, head_dim), gv)
    k = randn_bf16((tq, num_kv_heads, head_dim), gv)
    v = randn_bf16((tq, num_kv_heads, head_dim), gv)
    steps = [Step(StoreCall(k, v, meta.slot_mapping), PrefillCall(q, k, v, meta))]

    for s in range(1, extra_decode_steps + 1):
        lens = [L + s for L in seq_lens]
        tables = [bt[:num_blocks_for(L, block_size)] for bt, L in zip(tables_full, lens)]
        dm = decode_metadata(lens, tables, block_size)
        b = len(lens)
        qd = randn_bf16((b, num_heads, head_dim), gv)
        kd = randn_bf16((b, num_kv_heads, head_dim), gv)
        vd = randn_bf16((b, num_kv_heads, head_dim), gv)
        steps.append(Step(StoreCall(kd, vd, dm.slot_mapping), DecodeCall(qd, dm)))
    return Workload(name, num_heads, num_kv_heads, head_dim, block_size, num_blocks, steps, setup,
                    description=description)


def decode_workload(name: str, context_lens: list[int], num_heads: int, num_kv_heads: int,
                    head_dim: int, block_size: int, num_blocks: int, device="cpu",
                    description: str = "") -> Workload:
    """One decode step: every sequence already holds context_len - 1 tokens of
    N(0,1) history in the pool; the step stores the K/V of the token at
    position context_len - 1 and attends over all context_len tokens."""
    perm = torch.randperm(num_blocks, generator=generator(SEED_BLOCKS)).tolist()
    tables = _assign_blocks(perm, [num_blocks_for(L, block_size) for L in context_lens])
    hist_slots = []
    for bt, L in zip(tables, context_lens):
        hist_slots.extend(slots_of_positions(bt, range(L - 1), block_size))
    gv = generator(SEED_VALUES, device)
    t = len(hist_slots)
    hk = randn_bf16((t, num_kv_heads, head_dim), gv, device)
    hv = randn_bf16((t, num_kv_heads, head_dim), gv, device)
    dm = decode_metadata(context_lens, tables, block_size)
    b = len(context_lens)
    q = randn_bf16((b, num_heads, head_dim), gv, device)
    k = randn_bf16((b, num_kv_heads, head_dim), gv, device)
    v = randn_bf16((b, num_kv_heads, head_dim), gv, device)
    step = Step(StoreCall(k, v, dm.slot_mapping), DecodeCall(q, dm))
    return Workload(name, num_heads, num_kv_heads, head_dim, block_size, num_blocks, [step],
                    history_slots=torch.tensor(hist_slots, dtype=torch.int64),
                    history_k=hk, history_v=hv, description=description)


def mixed_workload(name: str, chunks: list[tuple[int, int]], decode_context_lens: list[int],
                   num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                   num_blocks: int, device="cpu", description: str = "") -> Workload:
    """One engine step that mixes chunked prefill and decode in a single varlen
    paged attention call.  ``chunks`` are (length after this step, tokens
    already in the cache) per prefilling sequence: the step queries the chunk
    cached .. length-1 (the boundary may fall inside a block).  Every decode
    sequence of context L queries its last token (q_len 1, L-1 cached).  All
    earlier tokens are history rows already in the pool; the step stores the
    new rows of every sequence, then attends.  Block tables are consecutive
    slices of one seeded permutation of the pool."""
    seqs = [(L, c) for L, c in chunks] + [(L, L - 1) for L in decode_context_lens]
    for L, c in seqs:
        if not 0 <= c < L:
            raise ValueError("every sequence needs at least one new token")
    perm = torch.randperm(num_blocks, generator=generator(SEED_BLOCKS)).tolist()
    tables = _assign_blocks(perm, [num_blocks_for(L, block_size) for L, _ in seqs])
    hist, new_slots, positions = [], [], []
    cu_q, cu_k = [0], [0]
    for (L, c), bt in zip(seqs, tables):
        hist.extend(slots_of_positions(bt, range(c), block_size))
        new_slots.extend(slots_of_positions(bt, range(c, L), block_size))
        positions.extend(range(c, L))
        cu_q.append(cu_q[-1] + L - c)
        cu_k.append(cu_k[-1] + L)
    meta = PrefillMeta(torch.tensor(cu_q, dtype=torch.int32), torch.tensor(cu_k, dtype=torch.int32),
                       max(L - c for L, c in seqs), max(L for L, _ in seqs),
                       torch.tensor(positions, dtype=torch.int64),
                       torch.tensor(new_slots, dtype=torch.int32), prepare_block_tables(tables))
    gv = generator(SEED_VALUES, device)
    t = len(hist)
    hk = randn_bf16((t, num_kv_heads, head_dim), gv, device)
    hv = randn_bf16((t, num_kv_heads, head_dim), gv, device)
    tq = cu_q[-1]
    q = randn_bf16((tq, num_heads, head_dim), gv, device)
    k = randn_bf16((tq, num_kv_heads, head_dim), gv, device)
    v = randn_bf16((tq, num_kv_heads, head_dim), gv, device)
    step = Step(StoreCall(k, v, meta.slot_mapping), PrefillCall(q, k, v, meta))
    return Workload(name, num_heads, num_kv_heads, head_dim, block_size, num_blocks, [step],
                    history_slots=torch.tensor(hist, dtype=torch.int64), history_k=hk, history_v=hv,
                    description=description)


def mixed_step_workload(device="cpu") -> Workload:
    """Mixed step on the Qwen3-8B attention shape (32/8/128, bs 256): four
    prompts in 1024-token chunks (first chunk of a 1024-token prompt; chunks
    1024..2047 and 2048..3071 of longer prompts; a 700-token tail after 1300
    cached, boundary inside a block) plus 128 decode rows with contexts
    ~ U[512, 4096]."""
    g = generator(SEED_LENGTHS)
    dec = torch.randint(512, 4097, (128,), generator=g).tolist()
    chunks = [(1024, 0), (2048, 1024), (3072, 2048), (2000, 1300)]
    need = sum(num_blocks_for(L, 256) for L, _ in chunks) + sum(num_blocks_for(L, 256) for L in dec)
    return mixed_workload("mixed_chunks_decode", chunks, dec, 32, 8, 128, 256, need + 64, device,
                          description="mixed: 4 prefill chunks (3772 tokens) + 128 decode rows "
                                      "ctx U[512,4096], 32/8/128 bs256")


# ---------------------------------------------------------------------------
# The five configurations of the hot path (attention shapes of Qwen3-0.6B:
# 16 query / 8 kv heads, and Qwen3-8B: 32 / 8 heads, head_dim 128).
# ---------------------------------------------------------------------------

def config1_tiny() -> Workload:
    """Tiny correctness case: Hq 2, Hkv 1, d 64, bs 16, 64-block pool; prompts of
    17 and 300 tokens (the second with its first 16 tokens cached), then 4
    decode steps on both."""
    return prefill_workload("tiny", [17, 300], [0, 1], 2, 1, 64, 16, 64, extra_decode_steps=4,
                            description="tiny: Hq2/Hkv1/d64 bs16 NB64, prompts 17 & 300 (16 cached), +4 decode")


def config2_decode(batch: int = 64, device="cpu") -> Workload:
    """Decode batch, Qwen3-0.6B attention shape: 64 sequences, context_lens
    uniform in [512, 4096], bs 256, blocks shuffled over a 2048-block pool."""
    ctx = torch.randint(512, 4097, (batch,), generator=generator(SEED_LENGTHS)).tolist()
    return decode_workload("decode_b64_qwen3_0.6b", ctx, 16, 8, 128, 256, 2048, device,
                           description="decode: B64 16/8/128 bs256 NB2048 ctx U[512,4096]")


def config3_prefill() -> Workload:
    """Varlen prefill with prefix cache, Qwen3-8B attention shape: 8 prompts
    uniform in [256, 2048], the first k in {0,1,2} full blocks cached (capped so
    that at least one token is queried), bs 256, 512-block pool."""
    g = generator(SEED_LENGTHS)
    lens = torch.randint(256, 2049, (8,), generator=g).tolist()
    ks = torch.randint(0, 3, (8,), generator=g).tolist()
    ks = [min(k, (L - 1) // 256) for k, L in zip(ks, lens)]
    return prefill_workload("prefill_b8_qwen3_8b", lens, ks, 32, 8, 128, 256, 512,
                            description="prefill: B8 32/8/128 bs256 NB512 L U[256,2048] prefix k in {0,1,2} blocks")


# 150 GB of K+V for one layer at 1 MiB per block (2 * 256 * 8 * 128 * 2 bytes).
CONFIG4_POOL_BLOCKS = 143051


def config4_context_lens(batch: int = 512) -> list[int]:
    g = generator(SEED_LENGTHS)
    short = torch.randint(128, 1025, (batch // 2,), generator=g)
    long_ = torch.randint(4096, 8193, (batch - batch // 2,), generator=g)
    both = torch.cat([short, long_])
    return both[torch.randperm(batch, generator=g)].tolist()


def config4_decode(num_blocks: int = CONFIG4_POOL_BLOCKS, batch: int = 512, device="cpu") -> Workload:
    """Large decode batch at max_num_seqs 512, Qwen3-8B attention shape, bs 256;
    context_lens half uniform in [128, 1024], half in [4096, 8192]; the pool is
    about 150 GB of K+V."""
    return decode_workload("decode_b512_qwen3_8b", config4_context_lens(batch), 32, 8, 128, 256,
                           num_blocks, device,
                           description=f"decode: B{batch} 32/8/128 bs256 NB{num_blocks} ctx 50% U[128,1024] + 50% U[4096,8192]")
