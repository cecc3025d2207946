"""Binding of the native block manager / scheduler (``include/kvpaged_sched.h``).

Argument marshalling only: the policy, the block manager and the metadata
builders run in the library's C++ code.  ``NativeScheduler.step()`` schedules
one engine step and returns the attention metadata for it, in the same form
as ``workloads.prefill_metadata`` / ``workloads.decode_metadata``.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _check, library
from .workloads import DecodeMeta, PrefillMeta

_P, _I32, _I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64

SIGNATURES = {
    "kvp_sched_create": (_P, [_I32, _I32, _I32, _I32]),
    "kvp_sched_destroy": (None, [_P]),
    "kvp_sched_add": (_I32, [_P, _I64, _P, _I32, _I32]),
    "kvp_sched_is_finished": (_I32, [_P]),
    "kvp_sched_schedule": (_I32, [_P, _P, _P]),
    "kvp_sched_step_sizes": (_I32, [_P, _P, _P]),
    "kvp_sched_prepare": (_I32, [_P, _P, _P, _P, _P, _P, _P, _I32, _P, _P, _P]),
    "kvp_sched_postprocess": (_I32, [_P, _P, _I32]),
    "kvp_sched_num_preemptions": (_I64, [_P]),
    "kvp_sched_num_free_blocks": (_I32, [_P]),
    "kvp_sched_seq_state": (_I32, [_P, _I64, _P, _P, _P, _P, _I32, _P]),
}


def _lib():
    lib = library()
    if not getattr(lib, "_kvp_sched_bound", False):
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype, f.argtypes = res, args
        lib._kvp_sched_bound = True
    return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class NativeScheduler:
    def __init__(self, num_blocks: int, block_size: int, max_num_seqs: int,
                 max_num_batched_tokens: int):
        self._lib = _lib()
        self._h = self._lib.kvp_sched_create(num_blocks, block_size, max_num_seqs,
                                             max_num_batched_tokens)
        if not self._h:
            _check(-1)
        self.block_size = block_size
        self.max_num_seqs = max_num_seqs
        self._ids = np.zeros(max_num_seqs, dtype=np.int64)
        self._ids_addr = self._ids.ctypes.data
        self._n = 0
        # out-parameters of the per-step calls, made once
        self._pre, self._t, self._mb = ctypes.c_int(), ctypes.c_int64(), ctypes.c_int()
        self._mq, self._mk, self._hp = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        self._refs = [ctypes.byref(x) for x in (self._pre, self._t, self._mb, self._mq, self._mk,
                                                 self._hp)]

    def close(self):
        if self._h:
            self._lib.kvp_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def add(self, seq_id: int, token_ids, max_tokens: int) -> None:
        t = np.ascontiguousarray(token_ids, dtype=np.int64)
        _check(self._lib.kvp_sched_add(self._h, seq_id, _p(t), t.shape[0], max_tokens))

    def is_finished(self) -> bool:
        return bool(self._lib.kvp_sched_is_finished(self._h))

    @property
    def num_preemptions(self) -> int:
        return int(self._lib.kvp_sched_num_preemptions(self._h))

    @property
    def num_free_blocks(self) -> int:
        return int(self._lib.kvp_sched_num_free_blocks(self._h))

    def seq_state(self, seq_id: int):
        nt, nc, st, ne = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        cap = 1 << 16
        table = np.zeros(cap, dtype=np.int32)
        _check(self._lib.kvp_sched_seq_state(self._h, seq_id, ctypes.byref(nt), ctypes.byref(nc),
                                             ctypes.byref(st), _p(table), cap, ctypes.byref(ne)))
        return {"num_tokens": nt.value, "num_cached_tokens": nc.value, "status": st.value,
                "block_table": table[:ne.value].tolist()}

    def step(self):
        """Schedules one step -> (seq_ids, is_prefill, metadata).  The int32
        metadata of a step shares one fresh buffer (the library fills every
        entry), so a step passes the library two addresses."""
        lib, h, r = self._lib, self._h, self._refs
        n = lib.kvp_sched_schedule(h, self._ids_addr, r[0])
        _check(min(n, 0))
        self._n = n
        _check(lib.kvp_sched_step_sizes(h, r[1], r[2]))
        T, MB = self._t.value, max(self._mb.value, 1)
        ids = self._ids[:n].tolist()
        pos = np.empty(T, dtype=np.int64)
        if self._pre.value:
            # [cu_q (n+1) | cu_k (n+1) | slots (T) | block tables (n x MB)]
            o1, o2, o3 = n + 1, 2 * (n + 1), 2 * (n + 1) + T
            buf = np.empty(o3 + n * MB, dtype=np.int32)
            b = buf.ctypes.data
            _check(lib.kvp_sched_prepare(h, b, b + 4 * o1, pos.ctypes.data, b + 4 * o2, None,
                                         b + 4 * o3, MB, r[3], r[4], r[5]))
            meta = PrefillMeta(torch.from_numpy(buf[:o1]), torch.from_numpy(buf[o1:o2]),
                               self._mq.value, self._mk.value, torch.from_numpy(pos),
                               torch.from_numpy(buf[o2:o3]),
                               torch.from_numpy(buf[o3:].reshape(n, MB)) if self._hp.value else None)
        else:
            # [context_lens (n) | slots (n) | block tables (n x MB)]
            buf = np.empty(2 * n + n * MB, dtype=np.int32)
            b = buf.ctypes.data
            _check(lib.kvp_sched_prepare(h, None, None, pos.ctypes.data, b + 4 * n, b, b + 8 * n,
                                         MB, None, None, None))
            ctx = buf[:n]
            meta = DecodeMeta(torch.from_numpy(pos), torch.from_numpy(ctx),
                              torch.from_numpy(buf[n:2 * n]),
                              torch.from_numpy(buf[2 * n:].reshape(n, MB)), int(ctx.max()))
        return ids, bool(self._pre.value), meta

    def postprocess(self, token_ids) -> None:
        t = np.ascontiguousarray(token_ids, dtype=np.int64)
        _check(self._lib.kvp_sched_postprocess(self._h, t.ctypes.data, t.shape[0]))
