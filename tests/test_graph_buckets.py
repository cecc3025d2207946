"""Bucket selection of the graph-replayed decode path (host logic, no GPU)."""
import pytest

from paged_kv_cache_125_gb300.graphs import bucket_for, default_buckets


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
