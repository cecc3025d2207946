"""Bucket selection of the graph-replayed decode path (host logic, no GPU)."""
import pytest

import torch

from paged_kv_cache_125_gb300.graphs import (bucket_for, default_buckets, pack_decode_metadata,
                                             packed_metadata_len)


def test_default_buckets_follow_the_pages_list():
    b = default_buckets(512)
    assert b[:5] == [1, 2, 4, 8, 16] and b[-1] == 512
    assert all(x % 16 == 0 for x in b[4:]) and len(b) == 4 + 32
    assert default_buckets(20) == [1, 2, 4, 8, 16, 20]
    assert default_buckets(3) == [1, 2, 3]


def test_bucket_for_picks_the_smallest_bucket_at_least_b():
    b = default_buckets(512)
    assert [bucket_for(b, n) for n in (1, 2, 3, 5, 9, 16, 17, 33, 500, 512)] == \
        [1, 2, 4, 8, 16, 16, 32, 48, 512, 512]
    with pytest.raises(ValueError):
        bucket_for(b, 513)


def test_packed_metadata_layout_and_padding():
    """[slot_mapping | context_lens | block_tables] for the bucket, padding rows
    slot -1 / context 0 / table -1, narrower tables padded with -1."""
    slots = torch.tensor([5, 300, 17], dtype=torch.int32)
    ctx = torch.tensor([6, 45, 18], dtype=torch.int32)
    bt = torch.tensor([[0, -1], [18, 7], [1, -1]], dtype=torch.int32)
    pb, width = 4, 3
    out = torch.full((packed_metadata_len(8, width),), 99, dtype=torch.int32)
    buf = pack_decode_metadata(pb, width, slots, bt, ctx, out=out)
    assert buf.numel() == packed_metadata_len(pb, width) == 4 * 5
    assert buf[:4].tolist() == [5, 300, 17, -1]
    assert buf[4:8].tolist() == [6, 45, 18, 0]
    assert buf[8:].view(4, 3).tolist() == [[0, -1, -1], [18, 7, -1], [1, -1, -1], [-1, -1, -1]]
    assert out[20:].eq(99).all()  # nothing written past the bucket's layout
    fresh = pack_decode_metadata(pb, width, slots, bt, ctx)
    assert torch.equal(fresh, buf)
    with pytest.raises(ValueError):
        pack_decode_metadata(2, width, slots, bt, ctx)  # more rows than the bucket
    with pytest.raises(ValueError):
        pack_decode_metadata(pb, 1, slots, bt, ctx)  # table wider than the graph's
