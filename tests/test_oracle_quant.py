"""Pins for the oracle's 8-bit quantized weight gather ("ZeRO Optimizer, in
depth", "Offload and ZeRO++"; "ZeRO and FSDP", "Fewer bytes on the wire"):
the rounding-error bound, the block maximum mapping to +-127, sign symmetry,
exact power-of-two scaling, ties to even, zero blocks and ragged blocks."""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(2025)


def _w(n, std=0.02):
    return oracle.cast_bf16((RNG.standard_normal(n) * std).astype(np.float32))


@pytest.mark.parametrize("block", [256, 512, 1024])
@pytest.mark.parametrize("n", [256, 1000, 4097, 65536])
def test_roundtrip_error_bound(block, n):
    w = _w(n)
    q, s = oracle.quantize_int8(w, block)
    back = oracle.bf16_to_f32(oracle.dequantize_int8(q, s, block)).astype(np.float64)
    x = oracle.bf16_to_f32(w).astype(np.float64)
    per = np.repeat(s.astype(np.float64), block)[:n]
    # half a quantization step plus half a bf16 ulp of the result
    bound = per / 2 * (1 + 1e-6) + np.abs(back) * 2.0 ** -8   # bf16 half-ulp <= 2^-8 relative
    assert np.all(np.abs(back - x) <= bound + 1e-45)
    assert q.min() >= -127 and q.max() <= 127


def test_block_max_maps_to_127_and_symmetry():
    n, block = 4096, 256
    w = _w(n)
    q, s = oracle.quantize_int8(w, block)
    x = oracle.bf16_to_f32(w).reshape(-1, block)
    qb = q.reshape(-1, block)
    for b in range(n // block):
        j = np.argmax(np.abs(x[b]))
        assert abs(int(qb[b, j])) == 127
        assert s[b] == np.float32(np.float32(np.abs(x[b]).max()) / np.float32(127.0))
    qn, sn = oracle.quantize_int8(w ^ np.uint16(0x8000), block)     # flip every sign
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(sn, s)


def test_power_of_two_scaling_is_exact():
    w = _w(3000)
    q, s = oracle.quantize_int8(w, 256)
    w8 = oracle.cast_bf16(oracle.bf16_to_f32(w) * np.float32(8.0))  # exact in bf16
    q8, s8 = oracle.quantize_int8(w8, 256)
    np.testing.assert_array_equal(q8, q)
    np.testing.assert_array_equal(s8, s * np.float32(8.0))


def test_ties_to_even_and_zero_blocks():
    # scale 1: values 127, 0.5, 1.5, 2.5, -2.5, 3.5 -> 127, 0, 2, 2, -2, 4
    vals = np.array([127.0, 0.5, 1.5, 2.5, -2.5, 3.5] + [0.0] * 250, np.float32)
    w = oracle.cast_bf16(np.concatenate([vals, np.zeros(256, np.float32)]))
    q, s = oracle.quantize_int8(w, 256)
    assert s[0] == np.float32(1.0) and s[1] == np.float32(0.0)
    np.testing.assert_array_equal(q[:6], [127, 0, 2, 2, -2, 4])
    assert not q[256:].any()
    back = oracle.dequantize_int8(q, s, 256)
    np.testing.assert_array_equal(back[256:], 0)


def test_ragged_last_block_and_wire_bytes():
    n, block = 1000, 256
    w = _w(n)
    q, s = oracle.quantize_int8(w, block)
    assert s.size == 4 and q.size == n
    x = oracle.bf16_to_f32(w)
    assert s[3] == np.float32(np.abs(x[768:]).max() / np.float32(127.0))
    # bytes a receiver gets per weight: 1 + 4/block, against 2 for bf16
    assert (q.nbytes + s.nbytes) / n == pytest.approx(1 + 4 * 4 / 1000)
    assert (1 + 4 / 256) / 2 == pytest.approx(0.5078125)
