"""CUDA-graph decode with batch-size buckets, the way the pages' engine runs
decode steps ("nano-vLLM-1", ModelRunner: graphs captured for batch sizes
1, 2, 4, 8, 16, 32, ... up to max_num_seqs; a step of b sequences replays the
graph of the smallest bucket >= b after copying its inputs into the graph's
fixed buffers; the unused rows are padding: slot_mapping -1, context_lens 0).

Every launch in a captured graph is a library call
(``attn_decode_paged_append``: the store of the new rows fused into the
paged decode); the launch configuration depends only on the bucket
and the fixed capacities, never on the step's data, so one capture serves
every step.  Padding rows write nothing (slot -1) and read nothing (context
0), and their output rows are zero.

Step metadata (slot_mapping, context_lens, block_tables) lives in one int32
buffer whose layout depends on the bucket pb (see ``pack_decode_metadata``):
each bucket's graph reads its own compact views of it, so a step's metadata,
padding rows included, arrives in ONE host-to-device copy of a packed pinned
buffer (``run_packed``).  q, k and v are not part of it: in an engine the
model's projections write them into the graph's fixed buffers.
"""
from __future__ import annotations

from . import attn_decode_paged_append, attn_decode_workspace_size


def default_buckets(max_bs: int) -> list[int]:
    """1, 2, 4, 8, then multiples of 16 up to max_bs (the pages' list)."""
    b = [x for x in (1, 2, 4, 8) if x <= max_bs]
    b += list(range(16, max_bs + 1, 16))
    if not b or b[-1] != max_bs:
        b.append(max_bs)
    return b


def packed_metadata_len(pb: int, width: int) -> int:
    """int32 entries of the packed metadata of bucket pb."""
    return pb * (2 + width)


def pack_decode_metadata(pb: int, width: int, slot_mapping, block_tables, context_lens, out=None):
    """Packs the metadata of a decode step of b = len(context_lens) <= pb
    sequences for the bucket-pb graph: ``[slot_mapping (pb) | context_lens (pb)
    | block_tables (pb x width)]`` int32, rows b .. pb-1 padded with slot -1,
    context 0 and block-table entries -1 (block-table columns past the
    caller's width are -1 as well).  ``out``: an int32 buffer of at least
    ``packed_metadata_len(pb, width)`` entries (pinned host memory for an
    asynchronous copy), else a new one on the host.  Returns the packed
    prefix of ``out``."""
    import torch
    b = int(context_lens.shape[0])
    if b > pb or slot_mapping.shape[0] != b or block_tables.shape[0] != b:
        raise ValueError("metadata rows must agree and fit the bucket")
    w = int(block_tables.shape[1])
    if w > width:
        raise ValueError("block table wider than the graph's width")
    n = packed_metadata_len(pb, width)
    if out is None:
        out = torch.empty((n,), dtype=torch.int32)
    buf = out[:n]
    buf[:pb].fill_(-1)
    buf[:b].copy_(slot_mapping)
    buf[pb:2 * pb].zero_()
    buf[pb:pb + b].copy_(context_lens)
    bt = buf[2 * pb:].view(pb, width)
    bt.fill_(-1)
    bt[:b, :w].copy_(block_tables)
    return buf


class _PackedMeta:
    """Per-bucket views of one int32 metadata buffer of max_bs x (2 + width)
    entries; bucket pb's views start at offset 0 in the packed layout."""

    def _init_meta(self, max_bs: int, width: int, dev) -> None:
        import torch
        self.width = width
        self.meta = torch.zeros((packed_metadata_len(max_bs, width),), dtype=torch.int32, device=dev)

    def meta_views(self, pb: int):
        """(slot_mapping, context_lens, block_tables) that bucket pb's graph reads."""
        m = self.meta
        return (m[:pb], m[pb:2 * pb],
                m[2 * pb:packed_metadata_len(pb, self.width)].view(pb, self.width))

    def _copy_meta(self, b: int, pb: int, slot_mapping, block_tables, context_lens) -> None:
        slots, ctx, bt = self.meta_views(pb)
        w = block_tables.shape[1]
        if w > self.width:
            raise ValueError("block table wider than max_blocks_per_seq")
        slots[:b].copy_(slot_mapping)
        bt[:b, :w].copy_(block_tables)
        ctx[:b].copy_(context_lens)
        if pb > b:  # padding rows: write nothing, read nothing
            slots[b:].fill_(-1)
            ctx[b:].fill_(0)

    def pack(self, b: int, slot_mapping, block_tables, context_lens, out=None):
        """Host-side packing of a step's metadata for this object's bucket of b."""
        return pack_decode_metadata(self.bucket(b), self.width, slot_mapping, block_tables,
                                    context_lens, out)

    def _load_packed(self, b: int, packed) -> int:
        pb = self.bucket(b)
        n = packed_metadata_len(pb, self.width)
        if packed.dtype != self.meta.dtype or packed.numel() < n:
            raise ValueError("packed metadata of the wrong type or size for this bucket")
        self.meta[:n].copy_(packed[:n], non_blocking=True)
        return pb


def bucket_for(buckets: list[int], b: int) -> int:
    """Smallest bucket >= b."""
    for x in buckets:
        if x >= b:
            return x
    raise ValueError(f"batch of {b} exceeds the largest bucket {buckets[-1]}")


class DecodeGraphs(_PackedMeta):
    """Captured store + decode graphs for one layer's cache.

    ``k_cache`` / ``v_cache``: [num_blocks, block_size, num_kv_heads, head_dim]
    bf16.  ``max_blocks_per_seq`` fixes the block-table width and the context
    capacity (max_blocks_per_seq * block_size) the graphs are planned for."""

    def __init__(self, k_cache, v_cache, num_heads: int, max_blocks_per_seq: int,
                 max_bs: int = 512, buckets: list[int] | None = None,
                 softmax_scale: float | None = None, stream=None):
        import torch
        self.k_cache, self.v_cache = k_cache, v_cache
        nb, bs, hkv, d = k_cache.shape
        dev = k_cache.device
        self.num_heads, self.num_kv_heads, self.head_dim, self.block_size = num_heads, hkv, d, bs
        self.max_bs = max_bs
        self.buckets = buckets or default_buckets(max_bs)
        if self.buckets[-1] > max_bs:
            raise ValueError("a bucket exceeds max_bs")
        self.capacity = max_blocks_per_seq * bs
        self.scale = softmax_scale if softmax_scale is not None else d ** -0.5
        bf16 = torch.bfloat16
        self.q = torch.zeros((max_bs, num_heads, d), dtype=bf16, device=dev)
        self.k = torch.zeros((max_bs, hkv, d), dtype=bf16, device=dev)
        self.v = torch.zeros((max_bs, hkv, d), dtype=bf16, device=dev)
        self._init_meta(max_bs, max_blocks_per_seq, dev)
        self.out = torch.zeros((max_bs, num_heads, d), dtype=bf16, device=dev)
        ws_bytes = attn_decode_workspace_size(max_bs, num_heads, d, self.capacity, bs)
        self.workspace = torch.empty((max(ws_bytes, 1),), dtype=torch.uint8, device=dev)
        self.stream = stream or torch.cuda.Stream(dev)
        self.graphs = {}
        for b in self.buckets:
            self.graphs[b] = self._capture(b)

    def _step(self, b: int) -> None:
        slots, ctx, bt = self.meta_views(b)
        attn_decode_paged_append(self.q[:b], self.k[:b], self.v[:b], slots, self.k_cache,
                                 self.v_cache, bt, ctx, self.capacity, softmax_scale=self.scale,
                                 workspace=self.workspace, out=self.out[:b])

    def _capture(self, b: int):
        import torch
        cur = torch.cuda.current_stream()
        self.stream.wait_stream(cur)
        with torch.cuda.stream(self.stream):
            self._step(b)  # warm-up outside the capture (library load, tensor maps)
        torch.cuda.current_stream().wait_stream(self.stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self._step(b)
        return g

    def bucket(self, b: int) -> int:
        return bucket_for(self.buckets, b)

    def run(self, q, k, v, slot_mapping, block_tables, context_lens):
        """One decode step of b = q.shape[0] sequences: store their new K/V rows
        at slot_mapping, attend over context_lens through block_tables.
        Returns a view of the first b output rows (valid until the next run)."""
        b = q.shape[0]
        pb = self.bucket(b)
        # No host read of context_lens (that would synchronise every step): a
        # context above the capacity is caught by the kernel, which skips the
        # row and sets KVP_ERR_DEVICE_DATA in the device status.
        self.q[:b].copy_(q)
        self.k[:b].copy_(k)
        self.v[:b].copy_(v)
        self._copy_meta(b, pb, slot_mapping, block_tables, context_lens)
        self.graphs[pb].replay()
        return self.out[:b]

    def run_packed(self, b: int, packed):
        """One decode step of b sequences whose new rows the caller has written
        into q/k/v[:b], with the step's metadata packed for bucket(b) by
        ``pack`` (one copy; from pinned host memory it is asynchronous, and the
        caller keeps the buffer unchanged until the copy has run).  Returns a
        view of the first b output rows (valid until the next run)."""
        pb = self._load_packed(b, packed)
        self.graphs[pb].replay()
        return self.out[:b]


class LayeredDecodeGraphs(_PackedMeta):
    """The decode step of a whole model as one graph per bucket: every layer's
    ``attn_decode_paged_append`` in one capture, the way the pages' engine
    captures its model forward for decode ("nano-vLLM-1", ModelRunner
    capture_cudagraph).

    ``kv_layers``: one (k_cache, v_cache) pair per layer, each
    [num_blocks, block_size, num_kv_heads, head_dim] bf16.  The caller writes
    each layer's new rows into ``q[l][:b]``, ``k[l][:b]``, ``v[l][:b]`` (fixed
    buffers) and passes the step's metadata, shared by all layers, to
    ``run``; layer l's output is ``out[l][:b]``.  The calls run one after the
    other on one stream, so they share one workspace."""

    def __init__(self, kv_layers, num_heads: int, max_blocks_per_seq: int, max_bs: int = 512,
                 buckets: list[int] | None = None, softmax_scale: float | None = None, stream=None):
        import torch
        self.kv_layers = list(kv_layers)
        nb, bs, hkv, d = self.kv_layers[0][0].shape
        dev = self.kv_layers[0][0].device
        n_layers = len(self.kv_layers)
        self.num_heads, self.num_kv_heads, self.head_dim, self.block_size = num_heads, hkv, d, bs
        self.max_bs = max_bs
        self.buckets = buckets or default_buckets(max_bs)
        if self.buckets[-1] > max_bs:
            raise ValueError("a bucket exceeds max_bs")
        self.capacity = max_blocks_per_seq * bs
        self.scale = softmax_scale if softmax_scale is not None else d ** -0.5
        bf16 = torch.bfloat16
        self.q = torch.zeros((n_layers, max_bs, num_heads, d), dtype=bf16, device=dev)
        self.k = torch.zeros((n_layers, max_bs, hkv, d), dtype=bf16, device=dev)
        self.v = torch.zeros((n_layers, max_bs, hkv, d), dtype=bf16, device=dev)
        self.out = torch.zeros((n_layers, max_bs, num_heads, d), dtype=bf16, device=dev)
        self._init_meta(max_bs, max_blocks_per_seq, dev)
        ws_bytes = attn_decode_workspace_size(max_bs, num_heads, d, self.capacity, bs)
        self.workspace = torch.empty((max(ws_bytes, 1),), dtype=torch.uint8, device=dev)
        self.stream = stream or torch.cuda.Stream(dev)
        self.graphs = {b: self._capture(b) for b in self.buckets}

    def _step(self, b: int) -> None:
        slots, ctx, bt = self.meta_views(b)
        for layer, (kc, vc) in enumerate(self.kv_layers):
            attn_decode_paged_append(self.q[layer, :b], self.k[layer, :b], self.v[layer, :b],
                                     slots, kc, vc, bt, ctx, self.capacity,
                                     softmax_scale=self.scale, workspace=self.workspace,
                                     out=self.out[layer, :b])

    def _capture(self, b: int):
        import torch
        cur = torch.cuda.current_stream()
        self.stream.wait_stream(cur)
        with torch.cuda.stream(self.stream):
            self._step(b)  # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(self.stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self._step(b)
        return g

    def bucket(self, b: int) -> int:
        return bucket_for(self.buckets, b)

    def run(self, b: int, slot_mapping, block_tables, context_lens) -> int:
        """One decode step of b sequences whose new rows the caller has written
        into q/k/v[:, :b]; returns the bucket replayed (outputs in out[:, :b])."""
        pb = self.bucket(b)
        self._copy_meta(b, pb, slot_mapping, block_tables, context_lens)
        self.graphs[pb].replay()
        return pb

    def run_packed(self, b: int, packed) -> int:
        """As ``run``, with the metadata packed for bucket(b) by ``pack`` and
        loaded in one copy; returns the bucket replayed."""
        pb = self._load_packed(b, packed)
        self.graphs[pb].replay()
        return pb
