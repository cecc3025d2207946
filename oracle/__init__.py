"""CPU reference oracle for paged KV-cache attention (fp64, scalar C).

TEST INFRASTRUCTURE ONLY.  This package is the checker: the test-suite, the
smoke check and the CPU-baseline leg of the benchmark are its only users.  The
CUDA library never imports, links or calls it, and it shares no code with the
library.  The arithmetic lives in ``oracle.c`` (see that file's header for the
pages each function follows); this module only compiles it (gcc, once) and
marshals arrays through ctypes.

Arrays: bf16 tensors are passed as their raw 16-bit patterns (``uint16``);
integer metadata as ``int32`` / ``int64``; outputs are fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_oracle(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(compile_oracle())
            p = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_kv_store.argtypes = [p, p, i64, i64, p, i64, p, p, i64, i32, i32, i32]
            lib.oracle_gather.argtypes = [p, i64, i32, i32, i32, p, i32, i64, p]
            lib.oracle_copy_blocks.argtypes = [p, i64, i64, i64, i64, p, i64]
            lib.oracle_prefill.argtypes = [p, i64, p, p, i64, p, p, i64, i32, p, i32, p, p,
                                           i32, i32, i32, i32, dbl, p, i64, p]
            lib.oracle_decode.argtypes = [p, i64, p, p, i64, i32, p, i32, p, i32, i32, i32,
                                          i32, dbl, p, i32, p]
            for f in (lib.oracle_kv_store, lib.oracle_gather, lib.oracle_copy_blocks, lib.oracle_prefill,
                      lib.oracle_decode, lib.oracle_num_threads):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _u16(t) -> np.ndarray:
    """bf16 torch tensor (CPU) or uint16 array -> C-contiguous uint16 numpy view."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16, t.dtype
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _arr(t, dtype) -> np.ndarray:
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(t, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def kv_store(k, v, slot_mapping, k_cache: np.ndarray, v_cache: np.ndarray) -> None:
    """Scatter rows of k, v ([N, Hkv, d] bf16) into the uint16 caches
    [NB, bs, Hkv, d] in place at slot_mapping (slot < 0 skipped)."""
    lib = _load()
    ku, vu = _u16(k), _u16(v)
    sm = _arr(slot_mapping, np.int32)
    nb, bs, hkv, d = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    n = sm.shape[0]
    _check(lib.oracle_kv_store(_ptr(ku), _ptr(vu), hkv * d, hkv * d, _ptr(sm), n,
                               _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d), "kv_store")


def gather(cache: np.ndarray, block_table_row, num_tokens: int) -> np.ndarray:
    """Tokens 0..num_tokens-1 of one sequence read through its block table ->
    uint16 [num_tokens, Hkv, d]."""
    lib = _load()
    nb, bs, hkv, d = cache.shape
    bt = _arr(block_table_row, np.int32)
    out = np.zeros((num_tokens, hkv, d), dtype=np.uint16)
    _check(lib.oracle_gather(_ptr(np.ascontiguousarray(cache)), nb, bs, hkv, d, _ptr(bt),
                             bt.shape[0], num_tokens, _ptr(out)), "gather")
    return out


def copy_blocks(kv_cache: np.ndarray, block_mapping) -> None:
    """Copy on write in place: kv_cache is uint16 [..., NB, bs, Hkv, d] (every
    leading index is one plane); block_mapping is [n, 2] (src, dst)."""
    lib = _load()
    assert kv_cache.dtype == np.uint16 and kv_cache.flags.c_contiguous
    nb = kv_cache.shape[-4]
    be = int(np.prod(kv_cache.shape[-3:]))
    planes = kv_cache.size // (nb * be)
    bm = _arr(block_mapping, np.int32).reshape(-1, 2)
    _check(lib.oracle_copy_blocks(_ptr(kv_cache), planes, nb * be, nb, be, _ptr(bm), bm.shape[0]),
           "copy_blocks")


def prefill(q, cu_seqlens_q, cu_seqlens_k, num_heads: int, num_kv_heads: int, scale: float,
            k=None, v=None, k_cache: np.ndarray | None = None, v_cache: np.ndarray | None = None,
            block_tables=None, rows=None) -> np.ndarray:
    """Varlen causal prefill -> fp64 [sum q, Hq, d].  Keys from the caches through
    block_tables when given, else from packed k, v.  ``rows`` restricts the
    computed packed query tokens (others stay 0)."""
    lib = _load()
    qu = _u16(q)
    total_q, hq, d = qu.shape
    assert hq == num_heads
    cq, ck = _arr(cu_seqlens_q, np.int32), _arr(cu_seqlens_k, np.int32)
    out = np.zeros((total_q, hq, d), dtype=np.float64)
    r = _arr(rows, np.int64)
    if block_tables is not None:
        bt = _arr(block_tables, np.int32)
        nb, bs = k_cache.shape[0], k_cache.shape[1]
        rc = lib.oracle_prefill(_ptr(qu), hq * d, None, None, 0, _ptr(k_cache), _ptr(v_cache),
                                nb, bs, _ptr(bt), bt.shape[1], _ptr(cq), _ptr(ck), cq.shape[0] - 1,
                                hq, num_kv_heads, d, scale, _ptr(r),
                                0 if r is None else r.shape[0], _ptr(out))
    else:
        ku, vu = _u16(k), _u16(v)
        rc = lib.oracle_prefill(_ptr(qu), hq * d, _ptr(ku), _ptr(vu), num_kv_heads * d, None, None,
                                0, 1, None, 0, _ptr(cq), _ptr(ck), cq.shape[0] - 1,
                                hq, num_kv_heads, d, scale, _ptr(r),
                                0 if r is None else r.shape[0], _ptr(out))
    _check(rc, "prefill")
    return out


def decode(q, k_cache: np.ndarray, v_cache: np.ndarray, block_tables, context_lens,
           num_heads: int, num_kv_heads: int, scale: float, seqs=None) -> np.ndarray:
    """Paged decode -> fp64 [B, Hq, d].  ``seqs`` restricts the computed
    sequences (others stay 0)."""
    lib = _load()
    qu = _u16(q)
    b, hq, d = qu.shape
    assert hq == num_heads
    bt = _arr(block_tables, np.int32)
    cl = _arr(context_lens, np.int32)
    s = _arr(seqs, np.int32)
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    out = np.zeros((b, hq, d), dtype=np.float64)
    _check(lib.oracle_decode(_ptr(qu), hq * d, _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(bt),
                             bt.shape[1], _ptr(cl), b, hq, num_kv_heads, d, scale, _ptr(s),
                             0 if s is None else s.shape[0], _ptr(out)), "decode")
    return out
