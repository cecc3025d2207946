"""GB300-native paged KV-cache attention: the data-parallel hot path of one
attention layer of a nano-vLLM-style serving engine.

Thin Python binding over the C ABI of ``libkvpaged.so`` (declared in
``include/kvpaged.h``).  Every function here only checks and marshals torch
tensors (device pointers, strides, the current CUDA stream) and calls the
library; all the work runs in the library's CUDA kernels.  There is no CPU or
PyTorch fallback: if the library cannot be loaded, every call raises.

    kv_store(k, v, slot_mapping, k_cache, v_cache)
    kv_copy_blocks(kv_cache, block_mapping)
    attn_prefill_varlen(q, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, ...)
    attn_prefill_varlen_append(q, k, v, slot_mapping, cu_seqlens_q, cu_seqlens_k, ...)
    attn_decode_paged(q, k_cache, v_cache, block_tables, context_lens, max_context_len, ...)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = ["kv_store", "kv_copy_blocks", "attn_prefill_varlen", "attn_prefill_varlen_append",
           "attn_mixed_step",
           "attn_decode_paged", "attn_decode_workspace_size", "attn_decode_paged_noalloc",
           "attn_decode_paged_append",
           "device_status", "selftest_wait", "library", "library_path", "KvpError"]

_LIB_LOCK = threading.Lock()
_LIB = None

KVP_OK = 0
ERROR_NAMES = {-1: "KVP_ERR_INVALID_ARG", -2: "KVP_ERR_UNSUPPORTED", -3: "KVP_ERR_WORKSPACE",
               -4: "KVP_ERR_CUDA", -5: "KVP_ERR_DEVICE_TIMEOUT", -6: "KVP_ERR_DEVICE_DATA"}

# Every symbol include/kvpaged.h declares, with its ctypes signature.
_P, _I64, _I32, _F32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "kvp_last_error": (ctypes.c_char_p, []),
    "kvp_version": (_I32, []),
    "kvp_device_status": (_I32, []),
    "kvp_selftest_wait": (_I32, [_I32, _P]),
    "kv_store": (_I32, [_P, _P, _I64, _I64, _P, _I64, _P, _P, _I64, _I32, _I32, _I32, _P]),
    "kv_copy_blocks": (_I32, [_P, _I64, _I64, _I64, _I64, _P, _I64, _P]),
    "attn_prefill_varlen": (_I32, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _P, _I64, _I32, _P, _I32,
                                   _P, _P, _I32, _I32, _I32, _P, _I32, _I32, _I32, _F32, _P, _I64,
                                   _P]),
    "attn_decode_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "attn_decode_paged": (_I32, [_P, _I64, _P, _P, _I64, _I32, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                 _I32, _F32, _P, _SZ, _P, _I64, _P]),
    "attn_decode_paged_noalloc": (_I32, [_P, _I64, _P, _P, _I64, _I32, _P, _I32, _P, _I32, _I32, _I32,
                                         _I32, _I32, _F32, _P, _I64, _P]),
    "attn_decode_paged_append": (_I32, [_P, _I64, _P, _P, _I64, _I64, _P, _P, _P, _I64, _I32, _P, _I32,
                                        _P, _I32, _I32, _I32, _I32, _I32, _F32, _P, _SZ, _P, _I64, _P]),
    "attn_prefill_varlen_append": (_I32, [_P, _I64, _I64, _P, _P, _I64, _P, _P, _P, _I64, _I32, _P, _I32,
                                          _P, _P, _I32, _I32, _I32, _P, _I32, _I32, _I32, _F32, _P, _I64,
                                          _P]),
    "attn_mixed_step": (_I32, [_P, _I64, _I64, _P, _P, _I64, _P, _P, _P, _I64, _I32, _P, _I32, _P, _P,
                               _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _SZ, _P, _I64,
                               _P]),
}


class KvpError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    from . import _build
    return _build.LIB


def library():
    """Loads libkvpaged.so (built by ``__graft_entry__.build()`` or
    ``python -m paged_kv_cache_125_gb300._build``).  Raises if it is missing."""
    global _LIB
    with _LIB_LOCK:
        if _LIB is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libkvpaged.so is not built ({path}); run "
                                   "`python -m paged_kv_cache_125_gb300._build` first")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype, f.argtypes = res, args
            _LIB = lib
    return _LIB


def _check(rc: int):
    if rc != KVP_OK:
        msg = library().kvp_last_error().decode(errors="replace")
        raise KvpError(rc, msg)


def _stream(t):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _require(t, name, dtype, ndim=None, device=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")


def _rows(t, name, heads, dim):
    """[tokens, heads, dim] with contiguous (heads, dim) -> row stride in elements."""
    if t.shape[1:] != (heads, dim):
        raise ValueError(f"{name} must be [*, {heads}, {dim}], got {tuple(t.shape)}")
    if t.stride(2) != 1 or t.stride(1) != dim:
        raise ValueError(f"{name}: each token row [heads, head_dim] must be contiguous")
    return t.stride(0)


def _cache_dims(k_cache, v_cache):
    import torch
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    _require(v_cache, "v_cache", torch.bfloat16, 4, k_cache.device)
    if k_cache.shape != v_cache.shape or not k_cache.is_contiguous() or not v_cache.is_contiguous():
        raise ValueError("k_cache / v_cache must be contiguous [num_blocks, block_size, kv_heads, head_dim]")
    return k_cache.shape


def device_status() -> int:
    """Reads and clears the device status word (synchronizes)."""
    return int(library().kvp_device_status())


def selftest_wait(arrive: bool, stream=None) -> None:
    """Launches the bounded-wait self-test on the current device: one thread
    waits 2 ms at most on a barrier that it arrives on first (arrive=True) or
    that nothing arrives on (the wait expires and KVP_ERR_DEVICE_TIMEOUT is
    recorded).  Read the outcome with device_status()."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(library().kvp_selftest_wait(1 if arrive else 0, ctypes.c_void_p(s.cuda_stream)))


def kv_store(k, v, slot_mapping, k_cache, v_cache) -> None:
    import torch
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache)
    _require(k, "k", torch.bfloat16, 3, k_cache.device)
    _require(v, "v", torch.bfloat16, 3, k_cache.device)
    _require(slot_mapping, "slot_mapping", torch.int32, 1, k_cache.device)
    n = slot_mapping.shape[0]
    if k.shape[0] != n or v.shape[0] != n or not slot_mapping.is_contiguous():
        raise ValueError("k, v, slot_mapping must agree on the token count")
    ks, vs = _rows(k, "k", hkv, d), _rows(v, "v", hkv, d)
    _check(library().kv_store(_ptr(k), _ptr(v), ks, vs, _ptr(slot_mapping), n, _ptr(k_cache),
                              _ptr(v_cache), nb, bs, hkv, d, _stream(k_cache)))


def kv_copy_blocks(kv_cache, block_mapping) -> None:
    """Copy-on-write block copies in every plane of ``kv_cache``.

    ``kv_cache`` is the engine's cache tensor ``[..., num_blocks, block_size,
    num_kv_heads, head_dim]`` (bf16, contiguous; every leading index, e.g. k/v
    and layer, is one plane).  ``block_mapping`` is ``[n, 2]`` int32 (src, dst)
    on the same device."""
    import torch
    if kv_cache.dtype != torch.bfloat16 or not kv_cache.is_cuda or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be a contiguous bf16 CUDA tensor")
    if kv_cache.dim() < 4:
        raise ValueError("kv_cache must be [..., num_blocks, block_size, num_kv_heads, head_dim]")
    _require(block_mapping, "block_mapping", torch.int32, 2, kv_cache.device)
    if block_mapping.shape[1] != 2 or not block_mapping.is_contiguous():
        raise ValueError("block_mapping must be a contiguous [n, 2] tensor")
    nb = kv_cache.shape[-4]
    block_elems = kv_cache.shape[-3] * kv_cache.shape[-2] * kv_cache.shape[-1]
    planes = kv_cache.numel() // (nb * block_elems)
    _check(library().kv_copy_blocks(_ptr(kv_cache), planes, nb * block_elems, nb, block_elems,
                                    _ptr(block_mapping), block_mapping.shape[0], _stream(kv_cache)))


def attn_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len, block_size) -> int:
    n = library().attn_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len, block_size)
    if n == 0 and num_seqs > 0:
        _check(-1)
    return int(n)


def attn_decode_paged(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                      softmax_scale: float | None = None, workspace=None, out=None):
    import torch
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache)
    dev = k_cache.device
    _require(q, "q", torch.bfloat16, 3, dev)
    b, hq = q.shape[0], q.shape[1]
    qs = _rows(q, "q", hq, d)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    if block_tables.shape[0] != b or context_lens.shape[0] != b:
        raise ValueError("block_tables / context_lens must have one row per sequence")
    if not block_tables.is_contiguous() or not context_lens.is_contiguous():
        raise ValueError("block_tables / context_lens must be contiguous")
    if out is None:
        out = torch.empty((b, hq, d), dtype=torch.bfloat16, device=dev)
    _require(out, "out", torch.bfloat16, 3, dev)
    os_ = _rows(out, "out", hq, d)
    need = attn_decode_workspace_size(b, hq, d, max_context_len, bs)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    _check(library().attn_decode_paged(
        _ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), b, int(max_context_len), hq, hkv, d, scale,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), os_,
        _stream(k_cache)))
    return out


def attn_decode_paged_append(q, k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens,
                             max_context_len: int, softmax_scale: float | None = None, workspace=None,
                             out=None):
    """kv_store(k, v, slot_mapping, k_cache, v_cache) followed by
    attn_decode_paged(q, ...), in one launch (see include/kvpaged.h).  Row b
    of k / v is sequence b's new token, stored at slot_mapping[b] (the slot
    of its position context_lens[b] - 1; -1 = padding row)."""
    import torch
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache)
    dev = k_cache.device
    _require(q, "q", torch.bfloat16, 3, dev)
    _require(k, "k", torch.bfloat16, 3, dev)
    _require(v, "v", torch.bfloat16, 3, dev)
    _require(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    b, hq = q.shape[0], q.shape[1]
    qs = _rows(q, "q", hq, d)
    ks, vs = _rows(k, "k", hkv, d), _rows(v, "v", hkv, d)
    if k.shape[0] != b or v.shape[0] != b or slot_mapping.shape[0] != b:
        raise ValueError("k, v and slot_mapping must have one row per sequence")
    if not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous")
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    if block_tables.shape[0] != b or context_lens.shape[0] != b:
        raise ValueError("block_tables / context_lens must have one row per sequence")
    if not block_tables.is_contiguous() or not context_lens.is_contiguous():
        raise ValueError("block_tables / context_lens must be contiguous")
    if out is None:
        out = torch.empty((b, hq, d), dtype=torch.bfloat16, device=dev)
    _require(out, "out", torch.bfloat16, 3, dev)
    os_ = _rows(out, "out", hq, d)
    need = attn_decode_workspace_size(b, hq, d, max_context_len, bs)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    _check(library().attn_decode_paged_append(
        _ptr(q), qs, _ptr(k), _ptr(v), ks, vs, _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), nb,
        bs, _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), b, int(max_context_len),
        hq, hkv, d, scale, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        os_, _stream(k_cache)))
    return out


def attn_decode_paged_noalloc(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                              out, softmax_scale: float | None = None):
    """attn_decode_paged without a workspace: the library's built-in scratch
    is used (see include/kvpaged.h for who needs this and its limits).  The
    caller passes ``out`` ([num_seqs, num_heads, head_dim] bf16): like the
    entry point, this wrapper allocates no device memory."""
    import torch
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache)
    dev = k_cache.device
    _require(q, "q", torch.bfloat16, 3, dev)
    b, hq = q.shape[0], q.shape[1]
    qs = _rows(q, "q", hq, d)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    if block_tables.shape[0] != b or context_lens.shape[0] != b:
        raise ValueError("block_tables / context_lens must have one row per sequence")
    if not block_tables.is_contiguous() or not context_lens.is_contiguous():
        raise ValueError("block_tables / context_lens must be contiguous")
    _require(out, "out", torch.bfloat16, 3, dev)
    if out.shape[0] != b:
        raise ValueError("out must have one row per sequence")
    os_ = _rows(out, "out", hq, d)
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    _check(library().attn_decode_paged_noalloc(
        _ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), b, int(max_context_len), hq, hkv, d, scale,
        _ptr(out), os_, _stream(k_cache)))
    return out


def attn_prefill_varlen(q, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                        k=None, v=None, k_cache=None, v_cache=None, block_tables=None,
                        num_kv_heads: int | None = None, positions=None,
                        softmax_scale: float | None = None, out=None):
    """Keys/values come from k_cache/v_cache through block_tables when block_tables
    is given (prefix-cache hit), else from the packed k, v rows."""
    import torch
    dev = q.device
    _require(q, "q", torch.bfloat16, 3)
    tq, hq, d = q.shape
    qs = _rows(q, "q", hq, d)
    _require(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, dev)
    _require(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1, dev)
    nseq = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != nseq + 1:
        raise ValueError("cu_seqlens_q / cu_seqlens_k lengths differ")
    if block_tables is not None:
        nb, bs, hkv, d2 = _cache_dims(k_cache, v_cache)
        if d2 != d:
            raise ValueError("head_dim of q and caches differ")
        _require(block_tables, "block_tables", torch.int32, 2, dev)
        if block_tables.shape[0] != nseq or not block_tables.is_contiguous():
            raise ValueError("block_tables must be contiguous [num_seqs, max_blocks]")
        kp = vp = None
        kvs = tk = 0
        kc, vc, mb = k_cache, v_cache, block_tables.shape[1]
    else:
        _require(k, "k", torch.bfloat16, 3, dev)
        _require(v, "v", torch.bfloat16, 3, dev)
        hkv = k.shape[1] if num_kv_heads is None else num_kv_heads
        kvs = _rows(k, "k", hkv, d)
        if _rows(v, "v", hkv, d) != kvs:
            raise ValueError("k and v must share a row stride")
        kp, vp, kc, vc, nb, bs, mb = k, v, None, None, 0, 16, 0
        tk = k.shape[0]
        if v.shape[0] != tk:
            raise ValueError("k and v must have the same number of rows")
    if out is None:
        out = torch.empty((tq, hq, d), dtype=torch.bfloat16, device=dev)
    _require(out, "out", torch.bfloat16, 3, dev)
    os_ = _rows(out, "out", hq, d)
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    _check(library().attn_prefill_varlen(
        _ptr(q), qs, tq, _ptr(kp), _ptr(vp), kvs, tk, _ptr(kc), _ptr(vc), nb, bs,
        _ptr(block_tables), mb,
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_seqlen_q), int(max_seqlen_k), nseq,
        _ptr(positions), hq, hkv, d, scale, _ptr(out), os_, _stream(q)))
    return out


def attn_prefill_varlen_append(q, k, v, slot_mapping, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                               max_seqlen_k: int, k_cache, v_cache, block_tables=None, positions=None,
                               softmax_scale: float | None = None, out=None):
    """kv_store(k, v, slot_mapping, k_cache, v_cache) followed by
    attn_prefill_varlen, in one launch (see include/kvpaged.h).  Row t of
    k / v is the new key / value of query row t; with block_tables the keys
    are read from the caches (paged), without them from k / v (packed, no
    cached prefix)."""
    import torch
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache)
    dev = k_cache.device
    _require(q, "q", torch.bfloat16, 3, dev)
    _require(k, "k", torch.bfloat16, 3, dev)
    _require(v, "v", torch.bfloat16, 3, dev)
    tq, hq = q.shape[0], q.shape[1]
    qs = _rows(q, "q", hq, d)
    kvs = _rows(k, "k", hkv, d)
    if _rows(v, "v", hkv, d) != kvs:
        raise ValueError("k and v must share a row stride")
    _require(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    if k.shape[0] != tq or v.shape[0] != tq or slot_mapping.shape[0] != tq or \
            not slot_mapping.is_contiguous():
        raise ValueError("k, v and slot_mapping must have one (contiguous) row per query row")
    _require(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, dev)
    _require(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1, dev)
    nseq = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != nseq + 1:
        raise ValueError("cu_seqlens_q / cu_seqlens_k lengths differ")
    mb = 0
    if block_tables is not None:
        _require(block_tables, "block_tables", torch.int32, 2, dev)
        if block_tables.shape[0] != nseq or not block_tables.is_contiguous():
            raise ValueError("block_tables must be contiguous [num_seqs, max_blocks]")
        mb = block_tables.shape[1]
    if out is None:
        out = torch.empty((tq, hq, d), dtype=torch.bfloat16, device=dev)
    _require(out, "out", torch.bfloat16, 3, dev)
    os_ = _rows(out, "out", hq, d)
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    _check(library().attn_prefill_varlen_append(
        _ptr(q), qs, tq, _ptr(k), _ptr(v), kvs, _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), nb,
        bs, _ptr(block_tables), mb, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_seqlen_q),
        int(max_seqlen_k), nseq, _ptr(positions), hq, hkv, d, scale, _ptr(out), os_, _stream(q)))
    return out


def attn_mixed_step(q, k, v, slot_mapping, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                    max_seqlen_k: int, k_cache, v_cache, block_tables, num_decode_seqs: int,
                    decode_sms: int = 0, softmax_scale: float | None = None, workspace=None, out=None):
    """A step of prefill chunks and decode rows (the last num_decode_seqs
    sequences, one query row each): kv_store of every new row, then the
    paged varlen prefill over all sequences, with the decode rows run by the
    decode kernel beside the chunks (see include/kvpaged.h)."""
    import torch
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache)
    dev = k_cache.device
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, name, torch.bfloat16, 3, dev)
    tq, hq = q.shape[0], q.shape[1]
    qs = _rows(q, "q", hq, d)
    kvs = _rows(k, "k", hkv, d)
    if _rows(v, "v", hkv, d) != kvs:
        raise ValueError("k and v must share a row stride")
    _require(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    if k.shape[0] != tq or v.shape[0] != tq or slot_mapping.shape[0] != tq or \
            not slot_mapping.is_contiguous():
        raise ValueError("k, v and slot_mapping must have one (contiguous) row per query row")
    _require(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, dev)
    _require(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1, dev)
    nseq = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != nseq + 1:
        raise ValueError("cu_seqlens_q / cu_seqlens_k lengths differ")
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    if block_tables.shape[0] != nseq or not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous [num_seqs, max_blocks]")
    if out is None:
        out = torch.empty((tq, hq, d), dtype=torch.bfloat16, device=dev)
    _require(out, "out", torch.bfloat16, 3, dev)
    os_ = _rows(out, "out", hq, d)
    need = attn_decode_workspace_size(max(num_decode_seqs, 1), hq, d, int(max_seqlen_k), bs)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    _check(library().attn_mixed_step(
        _ptr(q), qs, tq, _ptr(k), _ptr(v), kvs, _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), nb, bs,
        _ptr(block_tables), block_tables.shape[1], _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_seqlen_q),
        int(max_seqlen_k), nseq, int(num_decode_seqs), int(decode_sms), hq, hkv, d, scale, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), os_, _stream(q)))
    return out
