"""Host-side range logic of the step orchestration (no GPU): bucket ranges
intersected with an owned range, and their cut into pipeline pieces."""
import pytest

from zero_sharded_mixed_gb300 import step as zstep


def _covers(pieces, lo, hi):
    pos = lo
    for a, b in pieces:
        assert a == pos and b > a
        pos = b
    assert pos == hi


@pytest.mark.parametrize("N,n_dp,bucket", [(1_000_003, 4, 300_000), (77, 3, 8), (5000, 8, 10 ** 9)])
def test_bucket_ranges_cover_the_owned_range(zlib, N, n_dp, bucket):
    L = zlib.zero_layout([N], n_dp, bucket_elems=bucket)
    _covers(zstep.bucket_ranges(L), 0, L.padded_n)
    lo, hi = L.shard, 2 * L.shard
    r = zstep.bucket_ranges(L, lo, hi)
    _covers(r, lo, hi)
    assert all(a // L.bucket == (b - 1) // L.bucket for a, b in r)        # no range crosses a bucket


@pytest.mark.parametrize("chunk", [None, 8, 64, 1000, 10 ** 9])
def test_split_ranges(zlib, chunk):
    L = zlib.zero_layout([100_003], 3, bucket_elems=30_000)
    ranges = zstep.bucket_ranges(L)
    pieces = zstep.split_ranges(ranges, chunk)
    _covers(pieces, 0, L.padded_n)
    if chunk:
        assert all(b - a <= chunk for a, b in pieces)
        starts = {a for a, _ in ranges}
        assert all(a in starts or (a - max(s for s in starts if s <= a)) % chunk == 0 for a, _ in pieces)
    else:
        assert pieces == ranges
    with pytest.raises(ValueError):
        zstep.split_ranges(ranges, 12)
