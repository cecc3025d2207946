"""The algorithmic work the benchmark divides by, counted by hand on tiny
step metadata: causal FLOPs and bytes of a prefill layer call, bytes of a
decode layer call (no GPU)."""
import torch

from paged_kv_cache_125_gb300 import workloads as W
from paged_kv_cache_125_gb300.engine_replay import decode_bytes, prefill_flops, prefill_layer_bytes


def test_prefill_flops_causal_with_prefix():
    # sequence 0: 3 new tokens, no prefix -> rows see 1, 2, 3 keys; sequence 1:
    # 2 new tokens after 16 cached -> rows see 17, 18 keys
    m = W.prefill_metadata([3, 18], [0, 16], [[0], [1, 2]], 16)
    d, hq = 64, 4
    assert prefill_flops(m, d, hq) == 4 * d * hq * (1 + 2 + 3 + 17 + 18)


def test_prefill_layer_bytes():
    m = W.prefill_metadata([3, 18], [0, 16], [[0], [1, 2]], 16)
    hq, hkv, d = 4, 2, 64
    rows, cached = 3 + 2, 16
    q_and_out = rows * 2 * hq * d * 2
    new_rows_read_and_stored = rows * 2 * (2 * hkv * d * 2)
    prefix = cached * 2 * hkv * d * 2
    assert prefill_layer_bytes(m, hq, hkv, d) == q_and_out + new_rows_read_and_stored + prefix


def test_decode_bytes():
    ctx = [5, 17]
    m = W.decode_metadata(ctx, [[3], [4, 5]], 16)
    hq, hkv, d, bs = 4, 2, 64, 16
    row = hkv * d * 2
    expect = (4 * 2 * row                      # 2 new rows: read and stored, K and V
              + (5 + 17) * row * 2             # K and V of every context token
              + 2 * 2 * hq * d * 2             # q and out
              + (1 + 2) * 4 + 2 * 4)           # used block-table entries, context_lens
    assert decode_bytes(m, 2, hq, hkv, d, bs) == expect
