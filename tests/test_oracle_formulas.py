"""Pins for the oracle's memory and communication formulas: the numbers the pages print."""
import json
import math
import os

import numpy as np
import pytest

from oracle import formulas

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "memory_and_comm.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _round(x, decimals, half_up=False):
    if half_up:
        q = 10 ** decimals
        return math.floor(x * q + 0.5) / q
    return round(x, decimals)


@pytest.mark.parametrize("case", _golden()["memory"], ids=lambda c: c["source"][:60])
def test_memory_matches_printed_numbers(case):
    for stage, printed in case["stages"].items():
        got = formulas.zero_memory(case["N"], case["n_dp"], int(stage)) / case["unit"]
        assert _round(got, case["decimals"], case.get("round_half_up", False)) == printed, \
            (case["source"], stage, got, printed)


def test_free_memory_after_states():
    for case in _golden()["free_after_states"]:
        states = formulas.zero_memory(case["N"], case["n_dp"], case["stage"])
        free_gb = (case["gpu_bytes"] - states) / 1e9
        assert abs(free_gb - case["about_gb"]) <= case["within_gb"], (case["source"], free_gb)


def test_sixteen_bytes_per_parameter():
    g = _golden()["bytes_per_param"]
    assert g["weight16"] + g["grad16"] + g["master32"] + g["m32"] + g["v32"] == g["total"] == 16
    # plain data parallelism with one GPU holds exactly the 16 bytes per parameter
    assert formulas.zero_memory(1, 1, 0) == 16
    # the optimizer part is the K = 12 bytes: raising K by one adds N bytes at stage 0
    assert formulas.zero_memory(10, 1, 0, K=13) - formulas.zero_memory(10, 1, 0) == 10


def test_per_gpu_formulas_are_the_table():
    # the memory table of "ZeRO and FSDP": 16N, 4N + 12N/n, 2N + 14N/n, 16N/n
    for N in (1, 7, 1000, 7.5e9):
        for n in (1, 2, 3, 8, 64, 1000):
            assert formulas.zero_memory(N, n, 0) == pytest.approx(16 * N)
            assert formulas.zero_memory(N, n, 1) == pytest.approx(4 * N + 12 * N / n)
            assert formulas.zero_memory(N, n, 2) == pytest.approx(2 * N + 14 * N / n)
            assert formulas.zero_memory(N, n, 3) == pytest.approx(16 * N / n)


def test_stage_limits():
    lim = _golden()["limits"]
    N = 1e9
    huge = 10 ** 9
    assert formulas.zero_memory(N, huge, 1) / N == pytest.approx(lim["stage1_bytes_per_param_limit"], rel=1e-6)
    assert formulas.zero_memory(N, huge, 2) / N == pytest.approx(lim["stage2_bytes_per_param_limit"], rel=1e-6)
    assert 16 / (formulas.zero_memory(N, 64, 3) / N) == pytest.approx(lim["stage3_factor_at_64"])
    # memory never grows with the stage, and equals plain DP at n_dp = 1
    for n in (1, 2, 8, 64):
        mems = [formulas.zero_memory(N, n, s) for s in range(4)]
        assert mems == sorted(mems, reverse=True)
    assert len({formulas.zero_memory(N, 1, s) for s in range(4)}) == 1


@pytest.mark.parametrize("stage", [-1, 4, 5, "1", None, 1.5])
def test_invalid_stage_raises(stage):
    with pytest.raises(ValueError):
        formulas.zero_memory(10, 2, stage)
    with pytest.raises(ValueError):
        formulas.zero_comm_bytes(10, 2, stage)


def test_comm_stage12_equals_dp_and_stage3_is_one_and_a_half():
    for N in (1, 1000, 7e9):
        for n in (2, 3, 8, 128):
            dp = formulas.zero_comm_bytes(N, n, 0)
            assert formulas.zero_comm_bytes(N, n, 1) == pytest.approx(dp)
            assert formulas.zero_comm_bytes(N, n, 2) == pytest.approx(dp)
            assert formulas.zero_comm_bytes(N, n, 3) / dp == pytest.approx(1.5)


def test_comm_exact_ring_factor():
    # an all-reduce of N bf16 elements sends 2 (n-1)/n N elements per GPU
    assert formulas.zero_comm_bytes(8, 4, 0) == 2 * 3 / 4 * 8 * 2
    # one GPU sends nothing
    for s in range(4):
        assert formulas.zero_comm_bytes(1000, 1, s) == 0
    # as n grows the stage-0 volume tends to 2N elements, stage 3 to 3N
    N = 1e6
    assert formulas.zero_comm_bytes(N, 10 ** 9, 0, 1, 1) == pytest.approx(2 * N, rel=1e-6)
    assert formulas.zero_comm_bytes(N, 10 ** 9, 3, 1, 1) == pytest.approx(3 * N, rel=1e-6)


def test_comm_fp32_gradients_double_the_gradient_term():
    N, n = 1e9, 8
    for stage in (1, 2, 3):
        bf16 = formulas.zero_comm_bytes(N, n, stage, 2, 2)
        fp32g = formulas.zero_comm_bytes(N, n, stage, 2, 4)
        grad_term = (n - 1) / n * N * 2
        assert fp32g - bf16 == pytest.approx(grad_term)
    # stage 0 is all gradient: doubling its element size doubles it
    assert formulas.zero_comm_bytes(N, n, 0, 2, 4) == pytest.approx(2 * formulas.zero_comm_bytes(N, n, 0))
    # weights of a different size only change the weight term
    assert formulas.zero_comm_bytes(N, n, 0, 4, 2) == formulas.zero_comm_bytes(N, n, 0, 2, 2)


def test_comm_llama3_70b_printed():
    for case in _golden()["comm"]:
        if "gb" not in case:
            continue
        got = formulas.zero_comm_bytes(case["N"], case["n_dp"], case["stage"]) / 1e9
        assert got == pytest.approx(case["gb"], rel=case["rel_tol"]), (case["source"], got)


# The learning-rate schedule of the example configuration ("DeepSpeed ZeRO",
# "The configuration file": WarmupDecayLR with warmup_min_lr 0, warmup_max_lr
# 1e-4, warmup_num_steps 100, total_num_steps 10000), read as linear warmup
# then linear decay to 0, the first step at 0 schedule steps.
SCHED = dict(min_lr=0.0, max_lr=1e-4, warmup_steps=100, total_steps=10000)


def _lr(t, **kw):
    return formulas.warmup_decay_lr(t, **{**SCHED, **kw})


def test_schedule_points_of_the_example_configuration():
    f32 = lambda x: float(np.float32(x))
    assert _lr(1) == 0.0                   # the first step: warmup_min_lr
    assert _lr(51) == f32(5e-5)            # half way up
    assert _lr(101) == f32(1e-4)           # the end of warmup: warmup_max_lr
    assert _lr(5051) == f32(5e-5)          # half way down
    assert _lr(10001) == 0.0 and _lr(10_000_000) == 0.0   # 0 from total_num_steps on


def test_schedule_is_linear_in_each_phase():
    up = np.diff([_lr(t) for t in range(1, 102)])
    down = np.diff([_lr(t) for t in range(101, 10002)])
    assert np.allclose(up, 1e-6, rtol=1e-4)            # (1e-4 - 0) / 100 per step
    assert np.allclose(down, -1e-4 / 9900, rtol=2e-3)  # 1e-4 / (10000 - 100) per step
    assert (up > 0).all() and (down < 0).all()


def test_schedule_with_a_minimum_and_without_warmup():
    f32 = lambda x: float(np.float32(x))
    kw = dict(min_lr=1e-5, max_lr=1e-4, warmup_steps=10, total_steps=20)
    assert _lr(1, **kw) == f32(1e-5)
    assert _lr(6, **kw) == f32(1e-5 + 0.5 * 9e-5)    # half way up from the minimum
    assert _lr(16, **kw) == f32(5e-5)                 # half way down to 0, not to the minimum
    assert _lr(1, min_lr=1e-5, warmup_steps=0) == f32(1e-4)   # no warmup: the maximum at once


@pytest.mark.parametrize("bad", [dict(t=0), dict(warmup_steps=-1), dict(total_steps=100),
                                 dict(total_steps=50)])
def test_schedule_rejects_bad_parameters(bad):
    t = bad.pop("t", 1)
    with pytest.raises(ValueError):
        _lr(t, **bad)
