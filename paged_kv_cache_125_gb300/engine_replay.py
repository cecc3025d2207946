"""An engine's step loop over the attention hot path of every layer.

The loop an engine like the pages' runs ("nano-vLLM-1": Scheduler "2. prefill
的 schedule" / "3. decode 的 schedule", ModelRunner "4. prefill 输入打包",
"5. deocde 输入打包", "7. 性能优化"), reduced to its attention part:

* the native scheduler picks the step's sequences and builds the metadata;
* a prefill step is launched eagerly, one ``attn_prefill_varlen_append``
  per layer (the store of the step's new rows fused into the paged, or
  packed, varlen prefill);
* a decode step copies its packed metadata into the fixed buffer of a
  ``LayeredDecodeGraphs`` (one copy from pinned memory) and replays one graph
  that holds every layer's ``attn_decode_paged_append`` (store fused into the
  decode);
* the caller provides each step's per-layer q/k/v (an engine's projections)
  and the sampled tokens.

The benchmark times ``launch`` of this class and the GPU tests check its
outputs against the oracle, so both see the same calls.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _check, attn_prefill_varlen_append, library
from .graphs import LayeredDecodeGraphs
from .scheduler import NativeScheduler


@dataclass
class ReplayStep:
    seq_ids: list[int]
    is_prefill: bool
    meta: object          # workloads.PrefillMeta or workloads.DecodeMeta (host tensors)
    num_new: int          # new rows (= query rows) of the step
    dev: dict             # the step's metadata as the launch uses it (device copies / packed)


class EngineReplay:
    def __init__(self, requests, num_layers: int, num_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int, num_blocks: int, max_num_seqs: int, max_num_batched_tokens: int,
                 device, stream=None):
        """``requests``: (prompt token ids, max_tokens) pairs, submitted in order."""
        self.device = torch.device(device)
        self.num_layers, self.num_heads, self.num_kv_heads = num_layers, num_heads, num_kv_heads
        self.head_dim, self.block_size = head_dim, block_size
        self.scale = head_dim ** -0.5
        self.kv = torch.full((2, num_layers, num_blocks, block_size, num_kv_heads, head_dim),
                             float("nan"), dtype=torch.bfloat16, device=self.device)
        self.sched = NativeScheduler(num_blocks, block_size, max_num_seqs, max_num_batched_tokens)
        for i, (toks, out_len) in enumerate(requests):
            self.sched.add(i, toks, out_len)
        max_blocks = max((len(t) + o + block_size - 1) // block_size for t, o in requests)
        self.graphs = LayeredDecodeGraphs([(self.kv[0, l], self.kv[1, l]) for l in range(num_layers)],
                                          num_heads, max_blocks, max_bs=max_num_seqs,
                                          softmax_scale=self.scale, stream=stream)

    def done(self) -> bool:
        return self.sched.is_finished()

    @property
    def num_preemptions(self) -> int:
        return self.sched.num_preemptions

    def cache(self, layer: int):
        return self.kv[0, layer], self.kv[1, layer]

    def schedule(self) -> ReplayStep:
        """Schedules the next step and stages its metadata for the launch
        (prefill: asynchronous copies to the device; decode: packed for its
        bucket in pinned host memory)."""
        ids, pre, m = self.sched.step()
        dev = self.device
        if pre:
            n = int(m.cu_seqlens_q[-1])
            staged = {"slots": m.slot_mapping.to(dev, non_blocking=True),
                      "cu_q": m.cu_seqlens_q.to(dev, non_blocking=True),
                      "cu_k": m.cu_seqlens_k.to(dev, non_blocking=True),
                      "bt": None if m.block_tables is None else m.block_tables.to(dev, non_blocking=True)}
        else:
            n = len(ids)
            out = torch.empty((self.graphs.meta.numel(),), dtype=torch.int32, pin_memory=True)
            staged = {"packed": self.graphs.pack(n, m.slot_mapping, m.block_tables, m.context_lens, out=out)}
        return ReplayStep(ids, pre, m, n, staged)

    def decode_inputs(self, st: ReplayStep):
        """Views [layers, n, heads, d] of the graph buffers that a decode step's
        new q / k / v rows are written into before ``launch``."""
        n = st.num_new
        return self.graphs.q[:, :n], self.graphs.k[:, :n], self.graphs.v[:, :n]

    def launch(self, st: ReplayStep, q=None, k=None, v=None):
        """Launches the step on the current stream.  Prefill: q [layers, n, Hq,
        d], k / v [layers, n, Hkv, d] (layer l's new rows); returns the list of
        per-layer outputs.  Decode: the rows are already in ``decode_inputs``;
        returns the graph's output view [layers, n, Hq, d] (valid until the
        next decode step)."""
        if not st.is_prefill:
            self.graphs.run_packed(st.num_new, st.dev["packed"])
            return self.graphs.out[:, :st.num_new]
        return self._prefill(st, q, k, v)

    def _prefill(self, st: ReplayStep, q, k, v):
        """One attn_prefill_varlen_append per layer.  Layer 0 goes through the
        checked binding; the other layers reuse its marshalled arguments with
        the q / k / v / cache / out pointers moved by each tensor's layer
        stride (the tensors are [layers, ...] and contiguous)."""
        m, s = st.meta, st.dev
        for t in (q, k, v):
            if not t.is_contiguous() or t.shape[0] != self.num_layers:
                raise ValueError("prefill inputs must be contiguous [layers, rows, heads, head_dim]")
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=self.device)
        kc0, vc0 = self.kv[0, 0], self.kv[1, 0]
        attn_prefill_varlen_append(q[0], k[0], v[0], s["slots"], s["cu_q"], s["cu_k"], m.max_seqlen_q,
                                   m.max_seqlen_k, kc0, vc0, block_tables=s["bt"],
                                   softmax_scale=self.scale, out=out[0])
        if self.num_layers == 1:
            return [out[0]]
        nb, bs, hkv, d = kc0.shape
        n, hq = q.shape[1], q.shape[2]
        bt = s["bt"]
        stream = ctypes.c_void_p(torch.cuda.current_stream(self.device).cuda_stream)
        fn = library().attn_prefill_varlen_append
        qp, kp, vp, op = q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr()
        kcp, vcp = kc0.data_ptr(), vc0.data_ptr()
        sq, skv, so = q.stride(0) * 2, k.stride(0) * 2, out.stride(0) * 2
        scache = self.kv.stride(1) * 2
        fixed = (n, None, None, hkv * d, s["slots"].data_ptr(), None, None, nb, bs,
                 None if bt is None else bt.data_ptr(), 0 if bt is None else bt.shape[1],
                 s["cu_q"].data_ptr(), s["cu_k"].data_ptr(), m.max_seqlen_q, m.max_seqlen_k,
                 s["cu_q"].shape[0] - 1, None, hq, hkv, d, self.scale)
        for layer in range(1, self.num_layers):
            rc = fn(qp + layer * sq, hq * d, fixed[0], kp + layer * skv, vp + layer * skv, fixed[3],
                    fixed[4], kcp + layer * scache, vcp + layer * scache, *fixed[7:21],
                    op + layer * so, hq * d, stream)
            _check(rc)
        return [out[l] for l in range(self.num_layers)]

    def commit(self, st: ReplayStep, tokens) -> None:
        """The step's sampled tokens, one per scheduled sequence."""
        self.sched.postprocess(tokens)


def prefill_flops(meta, head_dim: int, num_heads: int) -> int:
    """Causal FLOPs of one prefill layer call: 4 * d * Hq * sum over queried
    rows of the keys each row sees (masked work excluded)."""
    ql = (meta.cu_seqlens_q[1:] - meta.cu_seqlens_q[:-1]).long()
    kl = (meta.cu_seqlens_k[1:] - meta.cu_seqlens_k[:-1]).long()
    return 4 * head_dim * num_heads * int((ql * (kl - ql) + ql * (ql + 1) // 2).sum())


def prefill_layer_bytes(meta, num_heads: int, num_kv_heads: int, head_dim: int) -> int:
    """Algorithmic bytes of one prefill layer call (store fused): q read and
    the output written (2 * Hq * d bf16 per query row), the new K/V rows read
    and stored (4 * Hkv * d bf16 per query row), and the cached prefix's K
    and V read once per kv head (2 * Hkv * d bf16 per cached key)."""
    ql = (meta.cu_seqlens_q[1:] - meta.cu_seqlens_q[:-1]).long()
    kl = (meta.cu_seqlens_k[1:] - meta.cu_seqlens_k[:-1]).long()
    rows, cached = int(ql.sum()), int((kl - ql).sum())
    return rows * (2 * num_heads + 4 * num_kv_heads) * head_dim * 2 + cached * 2 * num_kv_heads * head_dim * 2


def decode_bytes(meta, num_new: int, num_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int) -> int:
    """Algorithmic bytes of one decode layer call (store fused): the new rows
    read and written, K and V of every context token once per kv head, q and
    out, the used block-table entries and context_lens."""
    row = num_kv_heads * head_dim * 2
    c = meta.context_lens.long()
    return (4 * num_new * row + int(c.sum()) * row * 2 + 2 * num_new * num_heads * head_dim * 2 +
            int(((c + block_size - 1) // block_size).sum()) * 4 + num_new * 4)
