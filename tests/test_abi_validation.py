"""Host-side validation of the C ABI (no GPU): every call checks sizes,
supported shapes, strides, null pointers and alignment before it touches the
device, and reports the documented KVP_ERR_* code with a message.  The
pointers here are fake addresses that no case reaches a dereference of: each
case returns before the library's first CUDA call."""
import pytest

import paged_kv_cache_125_gb300 as kvp

OK, INVALID, UNSUPPORTED = 0, -1, -2
A = 0x10000          # a 16-byte aligned fake device address
MIS = 0x10002        # misaligned


@pytest.fixture(scope="module")
def lib():
    return kvp.library()


def _store(lib, **kw):
    a = dict(k=A, v=A, k_stride=8 * 128, v_stride=8 * 128, slots=A, n=4, kc=A, vc=A, nb=16, bs=256,
             hkv=8, d=128)
    a.update(kw)
    return lib.kv_store(a["k"], a["v"], a["k_stride"], a["v_stride"], a["slots"], a["n"], a["kc"],
                        a["vc"], a["nb"], a["bs"], a["hkv"], a["d"], None)


def _decode(lib, **kw):
    a = dict(q=A, q_stride=16 * 128, kc=A, vc=A, nb=64, bs=256, bt=A, mb=16, ctx=A, b=0, maxc=4096,
             hq=16, hkv=8, d=128, ws=A, ws_bytes=1 << 20, out=A, out_stride=16 * 128)
    a.update(kw)
    return lib.attn_decode_paged(a["q"], a["q_stride"], a["kc"], a["vc"], a["nb"], a["bs"], a["bt"],
                                 a["mb"], a["ctx"], a["b"], a["maxc"], a["hq"], a["hkv"], a["d"],
                                 0.088, a["ws"], a["ws_bytes"], a["out"], a["out_stride"], None)


def _prefill(lib, **kw):
    a = dict(q=A, q_stride=32 * 128, tq=0, k=None, v=None, kv_stride=8 * 128, tk=0, kc=A, vc=A,
             nb=64, bs=256, bt=A, mb=16, cq=A, ck=A, mq=0, mk=0, b=0, hq=32, hkv=8, d=128, out=A,
             out_stride=32 * 128)
    a.update(kw)
    return lib.attn_prefill_varlen(a["q"], a["q_stride"], a["tq"], a["k"], a["v"], a["kv_stride"],
                                   a["tk"], a["kc"], a["vc"], a["nb"], a["bs"], a["bt"], a["mb"],
                                   a["cq"], a["ck"], a["mq"], a["mk"], a["b"], None, a["hq"],
                                   a["hkv"], a["d"], 0.088, a["out"], a["out_stride"], None)


def _err(lib):
    return lib.kvp_last_error().decode()


def test_kv_store_validation(lib):
    assert _store(lib, n=0) == OK  # empty step: nothing to launch
    assert _store(lib, n=-1) == INVALID and "num_tokens" in _err(lib)
    assert _store(lib, hkv=0) == INVALID and "shape" in _err(lib)
    assert _store(lib, bs=0) == INVALID
    assert _store(lib, k_stride=8 * 128 - 1) == INVALID and "stride" in _err(lib)
    assert _store(lib, hkv=1 << 12, d=1 << 9, k_stride=1 << 21, v_stride=1 << 21) == UNSUPPORTED
    assert _store(lib, slots=None) == INVALID and "null" in _err(lib)
    assert _store(lib, kc=None) == INVALID


@pytest.mark.parametrize("hq,hkv,d,supported", [
    (16, 8, 128, True), (32, 8, 128, True), (8, 8, 128, True), (64, 8, 128, True),
    (16, 2, 64, True), (8, 1, 64, True),
    (24, 8, 128, False),  # G = 3
    (16, 16, 128, False),  # 16 kv heads
    (12, 3, 128, False),  # 3 kv heads
    (16, 8, 96, False),  # head_dim 96
    (128, 8, 128, False),  # G = 16
    (16, 0, 128, False),
])
def test_decode_supported_shapes(lib, hq, hkv, d, supported):
    rc = _decode(lib, hq=hq, hkv=hkv, d=d, q_stride=hq * d, out_stride=hq * d)
    assert rc == (OK if supported else UNSUPPORTED), _err(lib)


def test_decode_validation(lib):
    assert _decode(lib) == OK  # no sequences
    assert _decode(lib, b=-1) == INVALID and "bad sizes" in _err(lib)
    assert _decode(lib, nb=0) == INVALID
    assert _decode(lib, q_stride=16 * 128 - 8) == INVALID and "stride" in _err(lib)
    assert _decode(lib, mb=1 << 20, bs=4096) == UNSUPPORTED and "capacity" in _err(lib)
    assert _decode(lib, b=4, q=None) == INVALID and "null" in _err(lib)
    assert _decode(lib, b=4, ctx=None) == INVALID
    assert _decode(lib, b=4, q=MIS) == INVALID and "alignment" in _err(lib)
    assert _decode(lib, b=4, q_stride=16 * 128 + 4) == INVALID


@pytest.mark.parametrize("hq,hkv,d,bs,supported", [
    (32, 8, 128, 256, True), (16, 8, 128, 16, True), (64, 8, 128, 4096, True), (2, 1, 64, 16, True),
    (32, 16, 128, 256, True),  # any number of kv heads
    (32, 8, 128, 48, False),   # 3 x 16
    (32, 8, 128, 8, False),
    (32, 8, 128, 8192, False),
    (24, 8, 128, 256, False),  # G = 3
    (16, 1, 128, 256, False),  # G = 16
    (32, 8, 80, 256, False),
])
def test_prefill_supported_shapes(lib, hq, hkv, d, bs, supported):
    rc = _prefill(lib, hq=hq, hkv=hkv, d=d, bs=bs, q_stride=hq * d, out_stride=hq * d)
    assert rc == (OK if supported else UNSUPPORTED), _err(lib)


def test_prefill_validation(lib):
    assert _prefill(lib) == OK  # no sequences
    assert _prefill(lib, b=2, mq=16, tq=0) == OK  # nothing to query (every prompt cached)
    assert _prefill(lib, b=-1) == INVALID and "bad sizes" in _err(lib)
    assert _prefill(lib, q_stride=32 * 128 - 8) == INVALID and "stride" in _err(lib)
    live = dict(b=2, mq=16, mk=32, tq=20, tk=40)
    assert _prefill(lib, tq=1 << 31, **{k: v for k, v in live.items() if k != "tq"}) == INVALID
    assert _prefill(lib, cq=None, **live) == INVALID and "null" in _err(lib)
    assert _prefill(lib, kc=None, **live) == INVALID and "caches" in _err(lib)
    assert _prefill(lib, nb=1 << 20, bs=4096, **live) == UNSUPPORTED and "2^31" in _err(lib)
    assert _prefill(lib, kc=MIS, **live) == INVALID and "alignment" in _err(lib)
    assert _prefill(lib, bt=None, **live) == INVALID and "packed" in _err(lib)  # no k / v
    assert _prefill(lib, bt=None, k=A, v=A, kv_stride=8 * 128 + 4, **live) == INVALID
    assert _prefill(lib, q=MIS, **live) == INVALID and "alignment" in _err(lib)


def _copy(lib, **kw):
    a = dict(cache=A, planes=56, stride=160 * 256 * 8 * 128, nb=160, be=256 * 8 * 128, m=A, n=0)
    a.update(kw)
    return lib.kv_copy_blocks(a["cache"], a["planes"], a["stride"], a["nb"], a["be"], a["m"], a["n"],
                              None)


def test_copy_blocks_validation(lib):
    assert _copy(lib) == OK  # no pairs
    assert _copy(lib, n=-1) == INVALID and "num_pairs" in _err(lib)
    assert _copy(lib, planes=0) == INVALID and "shape" in _err(lib)
    assert _copy(lib, stride=160 * 256 * 8 * 128 - 1) == INVALID and "plane_stride" in _err(lib)
    assert _copy(lib, n=3, m=None) == INVALID and "null" in _err(lib)


def _append(lib, **kw):
    a = dict(q=A, qs=16 * 128, k=A, v=A, ks=8 * 128, vs=8 * 128, slots=A, kc=A, vc=A, nb=64, bs=256,
             bt=A, mb=16, ctx=A, b=0, maxc=4096, hq=16, hkv=8, d=128, ws=A, wsb=1 << 20, out=A,
             os=16 * 128)
    a.update(kw)
    return lib.attn_decode_paged_append(a["q"], a["qs"], a["k"], a["v"], a["ks"], a["vs"], a["slots"],
                                        a["kc"], a["vc"], a["nb"], a["bs"], a["bt"], a["mb"], a["ctx"],
                                        a["b"], a["maxc"], a["hq"], a["hkv"], a["d"], 0.088, a["ws"],
                                        a["wsb"], a["out"], a["os"], None)


def test_decode_append_validation(lib):
    assert _append(lib) == OK  # no sequences
    assert _append(lib, hq=64, qs=64 * 128, os=64 * 128) == OK  # eight heads per kv head, d 128
    assert _append(lib, b=-1) == INVALID and "bad sizes" in _err(lib)
    assert _append(lib, hkv=3, hq=12) == UNSUPPORTED and "unsupported" in _err(lib)
    assert _append(lib, ks=8 * 128 - 8) == INVALID and "stride" in _err(lib)
    assert _append(lib, mb=1 << 20, bs=4096) == UNSUPPORTED and "capacity" in _err(lib)
    assert _append(lib, nb=1 << 20, bs=4096, mb=16) == UNSUPPORTED and "2^31" in _err(lib)
    assert _append(lib, b=4, slots=None) == INVALID and "null" in _err(lib)
    assert _append(lib, b=4, k=MIS) == INVALID and "alignment" in _err(lib)
    assert _append(lib, b=4, vs=8 * 128 + 4) == INVALID


def _prefill_append(lib, **kw):
    a = dict(q=A, q_stride=32 * 128, tq=16, k=A, v=A, kv_stride=8 * 128, slots=A, kc=A, vc=A, nb=64,
             bs=256, bt=A, mb=16, cq=A, ck=A, mq=16, mk=16, b=1, hq=32, hkv=8, d=128, out=A,
             out_stride=32 * 128)
    a.update(kw)
    return lib.attn_prefill_varlen_append(a["q"], a["q_stride"], a["tq"], a["k"], a["v"], a["kv_stride"],
                                          a["slots"], a["kc"], a["vc"], a["nb"], a["bs"], a["bt"], a["mb"],
                                          a["cq"], a["ck"], a["mq"], a["mk"], a["b"], None, a["hq"],
                                          a["hkv"], a["d"], 0.088, a["out"], a["out_stride"], None)


def test_prefill_append_validation(lib):
    assert _prefill_append(lib, b=0) == OK            # no sequences: a no-op
    assert _prefill_append(lib, tq=0) == OK           # no query rows: a no-op
    assert _prefill_append(lib, b=-1) == INVALID and "bad sizes" in _err(lib)
    assert _prefill_append(lib, hq=24) == UNSUPPORTED and "attn_prefill_varlen_append" in _err(lib)
    assert _prefill_append(lib, bs=48) == UNSUPPORTED
    assert _prefill_append(lib, kv_stride=8 * 128 - 8) == INVALID and "stride" in _err(lib)
    assert _prefill_append(lib, nb=0) == INVALID and "num_blocks" in _err(lib)
    assert _prefill_append(lib, nb=1 << 24) == UNSUPPORTED and "2^31" in _err(lib)
    assert _prefill_append(lib, tq=-3) == INVALID and "total_q" in _err(lib)
    for name in ("q", "k", "v", "slots", "kc", "vc", "cq", "ck", "out"):
        assert _prefill_append(lib, **{name: None}) == INVALID and "null" in _err(lib), name
    assert _prefill_append(lib, mb=0) == INVALID and "max_blocks_per_seq" in _err(lib)
    for name in ("q", "k", "v", "kc", "vc", "out"):
        assert _prefill_append(lib, **{name: MIS}) == INVALID and "16-byte" in _err(lib), name
    assert _prefill_append(lib, kv_stride=8 * 128 + 4) == INVALID and "multiples of 8" in _err(lib)


def _mixed(lib, **kw):
    a = dict(q=A, q_stride=32 * 128, tq=20, k=A, v=A, kv_stride=8 * 128, slots=A, kc=A, vc=A, nb=64,
             bs=256, bt=A, mb=16, cq=A, ck=A, mq=16, mk=4096, b=5, nd=4, dsms=0, hq=32, hkv=8, d=128,
             ws=A, wsb=1 << 20, out=A, out_stride=32 * 128)
    a.update(kw)
    return lib.attn_mixed_step(a["q"], a["q_stride"], a["tq"], a["k"], a["v"], a["kv_stride"], a["slots"],
                               a["kc"], a["vc"], a["nb"], a["bs"], a["bt"], a["mb"], a["cq"], a["ck"],
                               a["mq"], a["mk"], a["b"], a["nd"], a["dsms"], a["hq"], a["hkv"], a["d"],
                               0.088, a["ws"], a["wsb"], a["out"], a["out_stride"], None)


def test_mixed_step_validation(lib):
    assert _mixed(lib, b=0, nd=0) == OK               # no sequences: a no-op
    assert _mixed(lib, tq=0, nd=0) == OK              # no query rows: a no-op
    assert _mixed(lib, nd=6) == INVALID and "bad sizes" in _err(lib)        # more decode rows than seqs
    assert _mixed(lib, nd=-1) == INVALID and "attn_mixed_step" in _err(lib)
    assert _mixed(lib, dsms=-1) == INVALID
    assert _mixed(lib, tq=3) == INVALID                # fewer query rows than decode rows
    assert _mixed(lib, tq=1 << 31) == INVALID
    assert _mixed(lib, hq=24) == UNSUPPORTED and "unsupported" in _err(lib)
    assert _mixed(lib, bs=48) == UNSUPPORTED
    assert _mixed(lib, hq=8, hkv=8, d=96) == UNSUPPORTED   # head_dim the decode does not take
    assert _mixed(lib, out_stride=32 * 128 - 8) == INVALID and "stride" in _err(lib)
    assert _mixed(lib, nb=0) == INVALID and "num_blocks" in _err(lib)
    assert _mixed(lib, nb=1 << 24) == UNSUPPORTED and "2^31" in _err(lib)
    assert _mixed(lib, mb=1 << 20, bs=4096, nb=16) == UNSUPPORTED and "capacity" in _err(lib)
    for name in ("q", "k", "v", "slots", "kc", "vc", "bt", "cq", "ck", "out"):
        assert _mixed(lib, **{name: None}) == INVALID and "null" in _err(lib), name
    for name in ("q", "k", "v", "kc", "vc", "out"):
        assert _mixed(lib, **{name: MIS}) == INVALID and "16-byte" in _err(lib), name
    assert _mixed(lib, q_stride=32 * 128 + 4) == INVALID and "multiples of 8" in _err(lib)
