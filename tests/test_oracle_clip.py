"""Pins for the oracle's clipping by the global gradient norm
("DeepSpeed ZeRO", "The configuration file": gradient_clipping 1.0):
torch.nn.utils.clip_grad_norm_ (a library routine with an fp32 norm),
numpy's fp64 sum of squares, the exactly rounded sum of the squares
(math.fsum), and closed forms."""
import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(99)


def test_norm_matches_numpy_fp64():
    for n_src, dtype in [(1, "f32"), (4, "f32"), (8, "bf16"), (3, "bf16")]:
        x = (RNG.standard_normal((n_src, 50_000)) * 1e-2).astype(np.float32)
        src = oracle.cast_bf16(x) if dtype == "bf16" else x
        g = oracle.reduce_mean(src, n_src).astype(np.float64)
        assert oracle.grad_norm_sq(src, n_src) == pytest.approx(float(np.sum(g * g)), rel=1e-12)


def test_norm_is_the_exact_sum_of_squares():
    """The squares of the fp32 mean are exact in fp64, so the norm's only
    rounding is the sum's: against the exactly rounded sum (math.fsum) it is
    within a few units in the last place, also for millions of terms, where a
    plain running fp64 sum drifts by about 1e-11."""
    for n_src, n, dtype, seed in [(3, 2_000_003, "bf16", 5), (8, 3_000_017, "bf16", 1), (2, 77_777, "f32", 4)]:
        x = (np.random.default_rng(seed).standard_normal((n_src, n)) * 1e-2).astype(np.float32)
        src = oracle.cast_bf16(x) if dtype == "bf16" else x
        g = oracle.reduce_mean(src, n_src).astype(np.float64)
        exact = math.fsum((g * g).tolist())
        assert oracle.grad_norm_sq(src, n_src) == pytest.approx(exact, rel=1e-15, abs=0)


@pytest.mark.parametrize("max_norm,scale", [(1.0, 1e-2), (1.0, 1.0), (0.5, 3e-3), (1.0, 1e-5)])
def test_clip_matches_torch(max_norm, scale):
    x = (RNG.standard_normal((4, 20_000)) * scale).astype(np.float32)
    g = oracle.reduce_mean(x, 4)
    ours = oracle.scale(g, oracle.clip_coef(oracle.grad_norm_sq(x, 4), max_norm))
    p = torch.nn.Parameter(torch.zeros(g.size))
    p.grad = torch.from_numpy(g.copy())
    torch.nn.utils.clip_grad_norm_([p], max_norm=max_norm, foreach=False)
    np.testing.assert_allclose(ours, p.grad.numpy(), rtol=1e-6, atol=0)
    # the clipped norm is max_norm when clipping is active, unchanged otherwise
    n_after = np.sqrt(np.sum(ours.astype(np.float64) ** 2))
    n_before = np.sqrt(np.sum(g.astype(np.float64) ** 2))
    assert n_after == pytest.approx(min(n_before, max_norm), rel=1e-5)


def test_closed_forms():
    # n equal values c: ||g|| = |c| sqrt(n) exactly when n is a square
    c, n = np.float32(0.03125), 10_000
    src = np.full((1, n), c, np.float32)
    assert oracle.grad_norm_sq(src, 1.0) == float(c) ** 2 * n
    coef = oracle.clip_coef(float(c) ** 2 * n, 1.0)
    assert coef == np.float32(1.0 / (float(c) * 100 + 1e-6))
    # below the threshold the coefficient is exactly 1 and scaling is the identity
    assert oracle.clip_coef(0.25, 1.0) == np.float32(1.0)
    g = (RNG.standard_normal(1000) * 1e-3).astype(np.float32)
    np.testing.assert_array_equal(oracle.scale(g, np.float32(1.0)), g)
    # a zero gradient has norm 0 and is left alone
    assert oracle.grad_norm_sq(np.zeros((2, 8), np.float32), 2.0) == 0.0
    assert oracle.clip_coef(0.0, 1.0) == np.float32(1.0)


def test_clip_then_adamw_first_step():
    # the first step from zero moments moves w by -lr * gc / (|gc| + eps), with
    # gc = coef * g the clipped mean gradient (closed form of the t = 1 step)
    hp = oracle.AdamW(lr=1e-3, weight_decay=0.0)
    x = (RNG.standard_normal((2, 4096)) * 10.0).astype(np.float32)
    w = np.zeros(4096, np.float32)
    z = np.zeros(4096, np.float32)
    nsq = oracle.grad_norm_sq(x, 2)
    coef = oracle.clip_coef(nsq, 1.0)
    assert coef < 1.0
    _, w_c, m_c, _ = oracle.rs_adamw_reference(x, 2, w, z, z, hp, 1, clip=(nsq, 1.0))
    gc = oracle.reduce_mean(x, 2).astype(np.float64) * float(coef)
    expect = -1e-3 * gc / (np.abs(gc) + float(np.float32(1e-8)))
    assert np.max(np.abs(w_c - expect)) <= 8 * np.spacing(np.float32(1e-3))
    # the first moment holds (1 - b1) times the clipped gradient
    np.testing.assert_allclose(m_c, 0.1 * gc, rtol=1e-6)
