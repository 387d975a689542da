"""Pins of the oracle's 8-bit gradient reduce-scatter (ZeRO++ quantized
gradients: "ZeRO Optimizer, in depth", "Offload and ZeRO++"; "ZeRO and FSDP",
"Fewer bytes on the wire").

Reading pinned here: each rank quantizes its gradient slice for owner o in
the weight gather's block format; blocks restart at every slice boundary; the
owner's value is code * scale rounded once to fp32; the mean over ranks is the
fp32 mean of the bf16 path.  What fixes it, without the oracle checking itself:

- gradients built from known codes and power-of-two steps quantize to exactly
  those codes and steps, dequantize to exactly the bf16 values, and then the
  whole 8-bit step equals the pinned bf16 step bit for bit (a wrong block,
  slice or rank scale, or a lost term, breaks the equality);
- on random gradients every value is within half a quantization step of the
  bf16 gradient (the error bound of round-to-nearest), and the mean within
  the mean of those half steps;
- each slice's first scale equals max|g| / 127 over that slice's first block,
  computed directly from the gradient."""
import numpy as np
import pytest

import oracle
from zero_sharded_mixed_gb300 import inputs

HP = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


def _exact_grads(n_src, n_dp, S, block, seed):
    """bf16 gradients j * c with known integer codes j (|j| <= 127, one |j| =
    127 per block) and a power-of-two step c per (rank, slice, block); one
    all-zero block per row.  Returns (g bits, codes, steps)."""
    rng = np.random.default_rng(seed)
    nb = -(-S // block)
    P = n_dp * S
    codes = rng.integers(-127, 128, size=(n_src, P)).astype(np.int8)
    steps = np.empty((n_src, n_dp * nb), dtype=np.float32)
    for r in range(n_src):
        for o in range(n_dp):
            for b in range(nb):
                lo = o * S + b * block
                hi = min(lo + block, (o + 1) * S)
                steps[r, o * nb + b] = np.float32(2.0 ** -(8 + (3 * r + 5 * o + 7 * b) % 13))
                codes[r, lo + int(rng.integers(0, hi - lo))] = 127 if rng.random() < 0.5 else -127
        zb = int(rng.integers(0, n_dp * nb))                      # one all-zero block
        o, b = divmod(zb, nb)
        lo = o * S + b * block
        codes[r, lo:min(lo + block, (o + 1) * S)] = 0
        steps[r, zb] = 0.0
    values = np.empty((n_src, P), dtype=np.float32)
    for r in range(n_src):
        for o in range(n_dp):
            k = np.arange(S)
            values[r, o * S:(o + 1) * S] = codes[r, o * S:(o + 1) * S].astype(np.float64) * \
                steps[r, o * nb + k // block].astype(np.float64)
    g = oracle.cast_bf16(values)
    assert np.array_equal(oracle.bf16_to_f32(g), values), "j * 2^-e must be a bf16 value"
    return g.reshape(n_src, P), codes, steps


@pytest.mark.parametrize("n_dp,S,block", [(4, 1000, 256), (3, 256, 256), (2, 2049, 512),
                                          (1, 300, 2048), (8, 777, 256)])
def test_exact_gradients_quantize_to_their_codes_and_step_like_bf16(n_dp, S, block):
    g, codes, steps = _exact_grads(n_dp, n_dp, S, block, seed=S + n_dp)
    q, scales = oracle.quantize_grad_int8(g, n_dp, block)
    assert np.array_equal(q, codes)
    assert np.array_equal(scales, steps)
    deq = oracle.dequantize_grad_int8(q, scales, n_dp, block)
    assert np.array_equal(deq, oracle.bf16_to_f32(g))
    P = n_dp * S
    w0 = inputs.master_weights(P, P, seed=1).numpy()
    z = np.zeros(P, np.float32)
    got = oracle.qgrad_rs_adamw_reference(q, scales, n_dp, block, n_dp, w0, z, z, HP, 1)
    ref = oracle.rs_adamw_reference(g, n_dp, w0, z, z, HP, 1)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("n_dp,S,block", [(4, 5000, 256), (8, 3001, 512), (3, 10_000, 2048)])
def test_error_within_half_a_step(n_dp, S, block):
    P = n_dp * S
    g = inputs.bf16_bits(inputs.grads_bf16(n_dp, P, P, seed=7, step=1, outlier_p=0.01))
    q, scales = oracle.quantize_grad_int8(g, n_dp, block)
    deq = oracle.dequantize_grad_int8(q, scales, n_dp, block).astype(np.float64)
    exact = oracle.bf16_to_f32(g).astype(np.float64)
    nb = -(-S // block)
    k = np.arange(P) % S
    o = np.arange(P) // S
    step = scales[:, o * nb + k // block].astype(np.float64)            # (n_src, P)
    # rounding to the nearest code: half a step; the fp32 product adds at most
    # half an fp32 ulp of |q| * step <= 127 * step
    bound = step * (0.5 + 127 * 2.0 ** -24) + 1e-45
    assert np.all(np.abs(deq - exact) <= bound)
    assert np.any(deq != exact)                                         # the bound is not vacuous
    mean_q = oracle.reduce_mean(deq.astype(np.float32), n_dp).astype(np.float64)
    mean_b = exact.sum(axis=0) / n_dp
    tol = bound.sum(axis=0) / n_dp + 4 * n_dp * 2.0 ** -24 * np.abs(deq).sum(axis=0) / n_dp
    assert np.all(np.abs(mean_q - mean_b) <= tol)


def test_blocks_restart_at_every_slice():
    """S = 300 with block 256: every slice has a 256-block and a 44-block; the
    slices' magnitudes differ by powers of ten, so each slice's scales come
    from that slice alone."""
    n_dp, S, block = 4, 300, 256
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.standard_normal(S) * 10.0 ** (-o) for o in range(n_dp)])
    g = oracle.cast_bf16(vals.astype(np.float32)).reshape(1, -1)
    _, scales = oracle.quantize_grad_int8(g, n_dp, block)
    x = oracle.bf16_to_f32(g)[0]
    for o in range(n_dp):
        first = np.abs(x[o * S:o * S + block]).max()
        last = np.abs(x[o * S + block:(o + 1) * S]).max()
        assert scales[0, 2 * o] == np.float32(first) / np.float32(127)
        assert scales[0, 2 * o + 1] == np.float32(last) / np.float32(127)


def test_exact_gradients_accumulate_like_bf16():
    """With exactly representable gradients the 8-bit accumulation equals the
    pinned bf16 accumulation (stage 2 and the stage-3 layer reduce-scatter),
    overwrite and add alike."""
    n_dp, S, block = 4, 600, 256
    g1, _, _ = _exact_grads(n_dp, n_dp, S, block, seed=11)
    g2, _, _ = _exact_grads(n_dp, n_dp, S, block, seed=12)
    q1, s1 = oracle.quantize_grad_int8(g1, n_dp, block)
    q2, s2 = oracle.quantize_grad_int8(g2, n_dp, block)
    a = oracle.accumulate_reduce_int8(None, q1, s1, n_dp, block, True)
    assert np.array_equal(a, oracle.accumulate_reduce(None, g1, True))
    a = oracle.accumulate_reduce_int8(a, q2, s2, n_dp, block, False)
    ref = oracle.accumulate_reduce(oracle.accumulate_reduce(None, g1, True), g2, False)
    assert np.array_equal(a, ref)


def test_first_micro_batch_overwrites_the_buffer():
    """With first set, a stale buffer is ignored: the result is the sum of the
    dequantized gradients alone, as for a fresh buffer and as the bf16
    accumulation (each window starts a new sum: "ZeRO and FSDP", the paragraph
    on gradient accumulation)."""
    n_dp, S, block = 3, 512, 256
    g, _, _ = _exact_grads(n_dp, n_dp, S, block, seed=21)
    q, s = oracle.quantize_grad_int8(g, n_dp, block)
    stale = np.random.default_rng(0).standard_normal(n_dp * S).astype(np.float32)
    fresh = oracle.accumulate_reduce_int8(None, q, s, n_dp, block, True)
    assert np.array_equal(oracle.accumulate_reduce_int8(stale, q, s, n_dp, block, True), fresh)
    assert np.array_equal(fresh, oracle.accumulate_reduce(stale, g, True))
