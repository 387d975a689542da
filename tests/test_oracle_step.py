"""Pins for the oracle's reduce-scatter, AdamW, ZeRO-1/2 step, accumulation and
gather, against things other than the oracle itself:

* torch.optim.AdamW (a library routine) for the n_dp = 1 special case;
* closed forms: the first step from zero moments, a constant gradient (the
  bias-corrected moments are then exactly g and g^2 at every step), a zero
  gradient (pure decay);
* exact arithmetic: dyadic gradients whose sums are exact in fp32, so the mean
  must equal the exact mean;
* the invariant that a ZeRO-1/2 step equals plain data parallelism
  ("ZeRO and FSDP", "The idea, one stage at a time": a ring all-reduce is a
  reduce-scatter followed by an all-gather);
* numpy's concatenation for the all-gather.
"""
import numpy as np
import pytest
import torch

import oracle

HP = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
RNG = np.random.default_rng(2024)


def _bf16(x):
    return oracle.cast_bf16(np.asarray(x, np.float32))


def _grads(n_dp, n, std=1e-3, rng=RNG):
    return _bf16(rng.standard_normal((n_dp, n)).astype(np.float32) * std)


def _dyadic_grads(n_dp, n, rng=RNG):
    # k * 2^-10 with |k| < 128: exact in bf16; sums of up to 2^16 of them are exact in fp32
    k = rng.integers(-127, 128, size=(n_dp, n)).astype(np.float32)
    return _bf16(k * np.float32(2.0 ** -10))


# ---------------------------------------------------------------- reduce-scatter

@pytest.mark.parametrize("n_dp", [1, 2, 4, 8, 16, 64])
def test_mean_is_exact_for_dyadic_power_of_two(n_dp):
    g = _dyadic_grads(n_dp, 4096)
    exact = oracle.bf16_to_f32(g).astype(np.float64).sum(axis=0) / n_dp
    got = oracle.reduce_mean(g, n_dp)
    np.testing.assert_array_equal(got.astype(np.float64), exact)


@pytest.mark.parametrize("n_dp", [3, 5, 7, 12])
def test_mean_is_one_rounding_of_exact_sum(n_dp):
    g = _dyadic_grads(n_dp, 4096)
    exact_sum = oracle.bf16_to_f32(g).astype(np.float64).sum(axis=0)
    # the sum is exact in fp32, so the mean is one IEEE division (numpy's, fp32)
    expect = exact_sum.astype(np.float32) / np.float32(n_dp)
    np.testing.assert_array_equal(oracle.reduce_mean(g, n_dp), expect)


@pytest.mark.parametrize("n_dp", [2, 3, 8, 16])
def test_mean_within_summation_bound(n_dp):
    g = _grads(n_dp, 1 << 14)
    x = oracle.bf16_to_f32(g).astype(np.float64)
    exact = x.sum(axis=0) / n_dp
    u = 2.0 ** -24
    bound = (n_dp * u / (1 - n_dp * u)) * np.abs(x).sum(axis=0) / n_dp + u * np.abs(exact)
    err = np.abs(oracle.reduce_mean(g, n_dp).astype(np.float64) - exact)
    assert np.all(err <= bound * 1.0000001 + 1e-45)


def test_mean_fp32_rows_and_order():
    # rows are added in ascending rank order, starting from +0: the result is the
    # left-to-right fp32 sum, which differs from another order on this input
    rows = np.array([[1.0], [2.0 ** -24], [2.0 ** -24]], dtype=np.float32)
    assert oracle.reduce_mean(rows, 1.0)[0] == np.float32(1.0)
    assert oracle.reduce_mean(rows[::-1].copy(), 1.0)[0] == np.float32(1.0) + np.float32(2.0 ** -23)
    # -0 + nothing else: +0 + -0 = +0
    assert np.signbit(oracle.reduce_mean(np.array([[-0.0]], np.float32), 1.0)[0]) == False  # noqa: E712


# ---------------------------------------------------------------- AdamW

def _torch_adamw(w0, grads_per_step, hp):
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False, fused=False)
    for g in grads_per_step:
        p.grad = torch.from_numpy(g.copy())
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def test_single_rank_matches_torch_adamw():
    n, steps = 1 << 14, 6
    w0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    gs = [(RNG.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(steps)]
    w, m, v = w0, np.zeros(n, np.float32), np.zeros(n, np.float32)
    # error carried from earlier steps shrinks by b1 each step; each step adds a
    # few roundings of the magnitudes of its two terms
    bound_m = np.zeros(n)
    for t, g in enumerate(gs, start=1):
        bound_m = 0.9 * bound_m + 1e-6 * (0.9 * np.abs(m) + 0.1 * np.abs(g))
        w, m, v = oracle.adamw(w, m, v, g, HP, t)
    tw, tm, tv = _torch_adamw(w0, gs, HP)
    # torch forms m by lerp and the denominator as sqrt(v)/sqrt(bc2): a few
    # roundings apart.  Bounds are relative to the magnitudes of the terms.
    assert np.all(np.abs(m - tm) <= bound_m + 1e-15)
    np.testing.assert_allclose(v, tv, rtol=1e-6, atol=0)
    np.testing.assert_allclose(w, tw, rtol=1e-6, atol=1e-9)


def test_first_step_closed_form():
    # from m = v = 0 the bias-corrected moments are g and g^2, so
    # w1 = w0 (1 - lr wd) - lr g / (|g| + eps) up to a few roundings
    n = 1 << 14
    w0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    g = (RNG.standard_normal(n) * 1e-3).astype(np.float32)
    w1, m1, v1 = oracle.adamw(w0, np.zeros(n, np.float32), np.zeros(n, np.float32), g, HP, 1)
    b1, b2 = np.float32(HP.beta1), np.float32(HP.beta2)
    np.testing.assert_array_equal(m1, (np.float32(1) - b1) * g)
    np.testing.assert_array_equal(v1, (np.float32(1) - b2) * (g * g))
    lr, wd, eps = (np.float64(x) for x in (HP.lr, HP.weight_decay, HP.eps))
    g64 = g.astype(np.float64)
    expect = w0.astype(np.float64) * (1 - lr * wd) - lr * g64 / (np.abs(g64) + eps)
    assert np.max(np.abs(w1 - expect)) <= 4 * np.spacing(np.float32(0.1))


def test_constant_gradient_closed_form():
    # with a constant gradient, m_t = (1 - b1^t) g and v_t = (1 - b2^t) g^2 exactly,
    # so every step moves w by lr g / (|g| + eps) after the decay
    n, steps = 4096, 25
    w = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    g = (RNG.choice([-1, 1], n) * (1e-3 + RNG.random(n) * 1e-3)).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    ref = w.astype(np.float64)
    lr, wd, eps = (np.float64(x) for x in (HP.lr, HP.weight_decay, HP.eps))
    g64 = g.astype(np.float64)
    for t in range(1, steps + 1):
        w, m, v = oracle.adamw(w, m, v, g, HP, t)
        ref = ref * (1 - lr * wd) - lr * g64 / (np.abs(g64) + eps)
        b1t = 1 - np.float64(np.float32(HP.beta1)) ** t
        np.testing.assert_allclose(m, b1t * g64, rtol=1e-5)
    assert np.max(np.abs(w - ref)) <= steps * 4 * np.spacing(np.float32(0.1))


def test_zero_gradient_is_pure_decay():
    n = 4096
    w0 = (RNG.standard_normal(n) * 0.02).astype(np.float32)
    z = np.zeros(n, np.float32)
    w, m, v = oracle.adamw(w0, z, z, z, HP, 1)
    np.testing.assert_array_equal(m, z)
    np.testing.assert_array_equal(v, z)
    lrwd = np.float32(HP.lr) * np.float32(HP.weight_decay)
    np.testing.assert_array_equal(w, w0 - lrwd * w0)


def test_bias_corrections():
    for t in (1, 2, 10, 1000, 10 ** 6):
        bc1, bc2 = oracle.bias_corrections(HP, t)
        b1 = np.float64(np.float32(0.9))
        b2 = np.float64(np.float32(0.999))
        assert bc1 == np.float32(1 - b1 ** t) and bc2 == np.float32(1 - b2 ** t)
    assert oracle.bias_corrections(HP, 1)[0] == np.float32(1) - np.float32(0.9)


# ---------------------------------------------------------------- ZeRO step

@pytest.mark.parametrize("n_dp,N,a", [(1, 100, 8), (2, 257, 8), (3, 1000, 1), (4, 4096, 8),
                                      (5, 333, 2), (8, 12345, 8), (16, 999, 8)])
def test_zero_step_equals_data_parallel(n_dp, N, a):
    L = oracle.layout([N], n_dp, align=a)
    S, P = L["shard"], L["padded"]
    w = np.zeros(P, np.float32)
    w[:N] = (RNG.standard_normal(N) * 0.02).astype(np.float32)
    m = np.zeros(P, np.float32)
    v = np.zeros(P, np.float32)
    w_dp, m_dp, v_dp = (np.tile(x, (n_dp, 1)) for x in (w, m, v))
    ws, ms, vs = (x.reshape(n_dp, S) for x in (w, m, v))
    for t in (1, 2, 3):
        g = np.zeros((n_dp, P), np.uint16)
        g[:, :N] = _grads(n_dp, N)
        full_z, ws, ms, vs = oracle.zero_step(g, ws, ms, vs, HP, t, n_copies=n_dp)
        full_d, w_dp, m_dp, v_dp = oracle.dp_step(g, w_dp, m_dp, v_dp, HP, t)
        # every rank ends with the same full weights as data parallelism
        np.testing.assert_array_equal(full_z, full_d)
        for r in range(n_dp):
            np.testing.assert_array_equal(ws.reshape(-1), w_dp[r])
            np.testing.assert_array_equal(ms.reshape(-1), m_dp[r])
            np.testing.assert_array_equal(vs.reshape(-1), v_dp[r])
        # the padding stays exactly zero
        assert not np.any(ws.reshape(-1)[N:]) and not np.any(full_z[:, N:])


def test_zero_step_does_not_modify_inputs_and_gathers_concatenation():
    n_dp, S = 4, 64
    g = _grads(n_dp, n_dp * S)
    ws = (RNG.standard_normal((n_dp, S)) * 0.02).astype(np.float32)
    ms = np.zeros((n_dp, S), np.float32)
    vs = np.zeros((n_dp, S), np.float32)
    copies = [x.copy() for x in (g, ws, ms, vs)]
    full, w2, m2, v2 = oracle.zero_step(g, ws, ms, vs, HP, 1, n_copies=2)
    for a, b in zip(copies, (g, ws, ms, vs)):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(full[0], np.concatenate([oracle.cast_bf16(w2[o]) for o in range(n_dp)]))
    np.testing.assert_array_equal(full[0], full[1])


def test_zero_step_shard_gets_its_own_gradient_piece():
    # lr = 0 keeps w, so m = (1-b1) * g exposes the gradient each rank received:
    # rank o's piece must be the data-parallel mean gradient on [o*S, (o+1)*S)
    n_dp, S = 4, 128
    g = _grads(n_dp, n_dp * S)
    hp0 = oracle.AdamW(lr=0.0, weight_decay=0.0)
    z = np.zeros((n_dp, S), np.float32)
    _, _, m, _ = oracle.zero_step(g, z, z, z, hp0, 1)
    gbar = oracle.reduce_mean(g, n_dp)
    np.testing.assert_array_equal(m.reshape(-1), (np.float32(1) - np.float32(0.9)) * gbar)


# ---------------------------------------------------------------- accumulation

def _accum_both_orders(micro, n_dp):
    """micro: list of K arrays (n_dp, P).  Returns (ZeRO-1 mean, ZeRO-2 mean)."""
    K = len(micro)
    acc = [None] * n_dp
    for k, g in enumerate(micro):
        for r in range(n_dp):
            acc[r] = oracle.accumulate_local(acc[r], g[r], first=(k == 0))
    z1 = oracle.reduce_mean(np.stack(acc), n_dp * K)
    A = None
    for k, g in enumerate(micro):
        A = oracle.accumulate_reduce(A, g, first=(k == 0))
    z2 = A / np.float32(n_dp * K)
    return z1, z2


def test_accumulation_orders_agree_exactly_on_dyadic_inputs():
    n_dp, K, P = 4, 4, 4096
    micro = [_dyadic_grads(n_dp, P) for _ in range(K)]
    z1, z2 = _accum_both_orders(micro, n_dp)
    exact = sum(oracle.bf16_to_f32(g).astype(np.float64).sum(axis=0) for g in micro) / (n_dp * K)
    np.testing.assert_array_equal(z1, z2)
    np.testing.assert_array_equal(z1.astype(np.float64), exact)


def test_accumulation_orders_within_summation_bound():
    n_dp, K, P = 4, 4, 1 << 14
    micro = [_grads(n_dp, P) for _ in range(K)]
    z1, z2 = _accum_both_orders(micro, n_dp)
    x = np.stack([oracle.bf16_to_f32(g).astype(np.float64) for g in micro])
    exact = x.sum(axis=(0, 1)) / (n_dp * K)
    nk, u = n_dp * K, 2.0 ** -24
    bound = nk * u / (1 - nk * u) * np.abs(x).sum(axis=(0, 1)) / nk + u * np.abs(exact)
    for z in (z1, z2):
        assert np.all(np.abs(z - exact) <= bound * 1.0000001 + 1e-45)


def test_first_micro_batch_overwrites_the_buffer():
    # "first" starts the window: whatever the buffer held before is replaced,
    # bit for bit, by this micro-batch's values (also the sign of zero)
    n_dp, n = 4, 1024
    g = _grads(n_dp, n)
    g[:, :4] = oracle.cast_bf16(np.array([-0.0, 0.0, -0.0, 1.0], np.float32))
    garbage = (RNG.standard_normal(n) * 1e3).astype(np.float32)
    acc = oracle.accumulate_local(garbage, g[0], first=True)
    np.testing.assert_array_equal(acc.view(np.uint32), oracle.bf16_to_f32(g[0]).view(np.uint32))
    A = oracle.accumulate_reduce(garbage, g, first=True)
    np.testing.assert_array_equal(A, oracle.accumulate_reduce(None, g, first=True))
    np.testing.assert_array_equal(A, oracle.reduce_mean(g, 1.0))
    # and an accumulating call adds onto what is there
    acc2 = oracle.accumulate_local(garbage, g[1], first=False)
    np.testing.assert_array_equal(acc2, garbage + oracle.bf16_to_f32(g[1]))


def test_single_micro_batch_accumulation_is_the_mean():
    n_dp, P = 8, 2048
    g = _grads(n_dp, P)
    A = oracle.accumulate_reduce(None, g, first=True)
    np.testing.assert_array_equal(A / np.float32(n_dp), oracle.reduce_mean(g, n_dp))
    acc = oracle.accumulate_local(None, g[3], first=True)
    np.testing.assert_array_equal(acc, oracle.bf16_to_f32(g[3]))


# ---------------------------------------------------------------- gather

def test_all_gather_is_concatenation():
    for n_dp, S in [(1, 8), (3, 5), (8, 1000)]:
        shards = RNG.integers(0, 1 << 16, size=(n_dp, S)).astype(np.uint16)
        np.testing.assert_array_equal(oracle.all_gather(shards), np.concatenate(list(shards)))
