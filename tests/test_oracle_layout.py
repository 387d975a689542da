"""Pins for the oracle's layout: brute force over small sizes, the properties the
pages fix (equal contiguous shards covering the flat vector, rank r owns shard
r), and the element counts of the two model shapes used by the workloads."""
import itertools

import numpy as np
import pytest

import oracle
from zero_sharded_mixed_gb300 import inputs


def _brute_shard(N, n_dp, a):
    # the smallest multiple of a whose n_dp copies hold all N elements
    s = 0
    while s * n_dp < N:
        s += a
    return s


@pytest.mark.parametrize("a", [1, 2, 8, 64])
def test_brute_force_small(a):
    for N in range(0, 301):
        for n_dp in range(1, 17):
            L = oracle.layout([N], n_dp, align=a, bucket=1)
            S, P = L["shard"], L["padded"]
            assert L["n"] == N
            assert S == _brute_shard(N, n_dp, a)
            assert S % a == 0 and P == n_dp * S
            assert 0 <= P - N < n_dp * a
            # shards [r*S, (r+1)*S) are contiguous, disjoint and cover [0, P)
            owner = np.repeat(np.arange(n_dp), S)
            assert owner.size == P and np.all(np.diff(owner) >= 0)


def test_offsets_are_prefix_sums_without_gaps():
    rng = np.random.default_rng(3)
    for _ in range(200):
        numels = rng.integers(0, 50, size=rng.integers(0, 12)).tolist()
        L = oracle.layout(numels, 3, align=8, bucket=16)
        expect = np.concatenate([[0], np.cumsum(numels)[:-1]]) if numels else np.zeros(0)
        np.testing.assert_array_equal(L["offsets"], expect.astype(np.int64))
        assert L["n"] == sum(numels)


def test_buckets_cover_the_padded_vector():
    for P_target, B, a in itertools.product([0, 1, 7, 64, 1000], [1, 3, 8, 100, 5000], [1, 8]):
        L = oracle.layout([P_target], 1, align=a, bucket=B)
        bq, nb, P = L["bucket"], L["n_buckets"], L["padded"]
        assert bq % a == 0 and bq >= B and bq - B < a
        assert nb == -(-P // bq)
        ranges = [(b * bq, min((b + 1) * bq, P)) for b in range(nb)]
        covered = sum(e - s for s, e in ranges)
        assert covered == P
        assert all(s < e for s, e in ranges)


@pytest.mark.parametrize("kw", [dict(n_dp=0), dict(n_dp=-1), dict(align=0), dict(bucket=0)])
def test_invalid_arguments(kw):
    args = dict(n_dp=2, align=8, bucket=8)
    args.update(kw)
    with pytest.raises(ValueError):
        oracle.layout([10], **args)


def test_negative_numel_and_overflow():
    with pytest.raises(ValueError):
        oracle.layout([5, -1], 2)
    with pytest.raises(ValueError):
        oracle.layout([2 ** 62, 2 ** 62], 2)


def test_model_shapes():
    gpt = inputs.gpt2xl_numels()
    assert sum(gpt) == 1_557_611_200
    assert len(gpt) == 2 + 48 * 12 + 2
    llama = inputs.llama7b_numels()
    assert sum(llama) == 6_738_415_616
    units = inputs.llama7b_units()
    assert len(units) == 34 and sum(units[1]) == 202_383_360
    assert sum(units[0]) == 131_072_000 and sum(units[-1]) == 131_076_096


def test_workload_layouts():
    # GPT-2 XL at n_dp = 8 with 5e8-element buckets: no padding, 4 buckets
    L = oracle.layout(inputs.gpt2xl_numels(), 8, align=8, bucket=500_000_000)
    assert (L["shard"], L["padded"], L["n_buckets"]) == (194_701_400, 1_557_611_200, 4)
    # the same at n_dp = 4
    L = oracle.layout(inputs.gpt2xl_numels(), 4)
    assert (L["shard"], L["padded"]) == (389_402_800, 1_557_611_200)
    # Llama-7B at n_dp = 8: one owned shard is 842,301,952 elements
    L = oracle.layout(inputs.llama7b_numels(), 8)
    assert (L["shard"], L["padded"]) == (842_301_952, 6_738_415_616)
    # the tiny config: N = 2^20 at n_dp = 4
    L = oracle.layout([1 << 20], 4)
    assert (L["shard"], L["padded"], L["n_buckets"]) == (262_144, 1 << 20, 1)
