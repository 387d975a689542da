"""Pins for the oracle's bf16 conversions against torch's own bf16 conversion
(a library routine), on special values, every tie pattern of a few upper
halves, and a few million random bit patterns."""
import numpy as np
import pytest
import torch

import oracle


def _torch_rne(x_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _is_nan_bf16(h):
    h = np.asarray(h, np.uint16)
    return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)


def _check(bits_u32: np.ndarray):
    x = bits_u32.astype(np.uint32).view(np.float32)
    ours = oracle.cast_bf16(x)
    ref = _torch_rne(x)
    nan_in = np.isnan(x)
    # NaN stays NaN (payload is not part of the contract)
    assert np.all(_is_nan_bf16(ours[nan_in]))
    # NaN keeps its sign
    assert np.array_equal(ours[nan_in] >> 15, (bits_u32[nan_in] >> 31).astype(np.uint16))
    np.testing.assert_array_equal(ours[~nan_in], ref[~nan_in])


def test_special_values():
    specials = np.array([
        0x00000000, 0x80000000,             # +-0
        0x7F800000, 0xFF800000,             # +-inf
        0x7FC00000, 0xFFC00000, 0x7F800001, 0xFFBFFFFF,  # NaNs (quiet, signalling)
        0x7F7FFFFF, 0xFF7FFFFF,             # largest finite -> rounds to inf
        0x7F7F7FFF, 0x7F7F8000, 0x7F7F8001,  # just below / at / above the overflow tie
        0x00800000, 0x00000001, 0x007FFFFF, 0x80000001,  # min normal, denormals
        0x3F808000, 0x3F818000,             # ties at 1.0: to even down, to even up
        0x3F807FFF, 0x3F808001,             # just below / above the tie
    ], dtype=np.uint32)
    _check(specials)


def test_every_low_half_for_some_upper_halves():
    uppers = np.array([0x0000, 0x0001, 0x007F, 0x0080, 0x3F80, 0x3F81, 0x4049, 0x7F7E, 0x7F7F,
                       0x8000, 0xBF80, 0xFF7F, 0xC2F6], dtype=np.uint32)
    low = np.arange(1 << 16, dtype=np.uint32)
    bits = (uppers[:, None] << 16 | low[None, :]).reshape(-1)
    _check(bits)


def test_random_bit_patterns():
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    _check(bits)


def test_random_normal_values():
    rng = np.random.default_rng(7)
    for scale in (1e-3, 0.02, 1.0, 1e30, 1e-38):
        x = (rng.standard_normal(1 << 18) * scale).astype(np.float32)
        _check(x.view(np.uint32))


def test_widen_is_exact():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f32(h)
    t = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    nan = np.isnan(t)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan].view(np.uint32), t[~nan].view(np.uint32))
    # round trip: widening then rounding gives back every non-NaN pattern
    back = oracle.cast_bf16(ours)
    np.testing.assert_array_equal(back[~nan], h[~nan])
    # scalar entry points agree with the array ones
    lib = oracle._load()
    for v in (0x3F80, 0xC2F6, 0x0001, 0x7F7F):
        assert lib.oracle_bf16_to_f32(v) == float(oracle.bf16_to_f32(np.uint16(v)))
        assert lib.oracle_f32_to_bf16(float(oracle.bf16_to_f32(np.uint16(v)))) == v


@pytest.mark.parametrize("value,expected", [
    (1.0, 0x3F80),
    (1.0 + 2 ** -8, 0x3F80),          # tie between 1 and 1+2^-7, even is 1
    (1.0 + 3 * 2 ** -8, 0x3F82),      # tie, even neighbour is above
    (-2.0, 0xC000),
    (3.0e38, 0x7F62),
])
def test_worked_values(value, expected):
    assert int(oracle.cast_bf16(np.array([value], np.float32))[0]) == expected


def test_quiet_nan_payload_survives_a_widening_round_trip():
    """IEEE 754-2019, 6.2.3: a quiet NaN converted to a wider format and back
    keeps its payload.  Every quiet bf16 NaN pattern of both signs, widened
    exactly to fp32 (its bits in the upper half), must come back unchanged."""
    quiet = np.array([h for h in range(1 << 16) if (h & 0x7FC0) == 0x7FC0], dtype=np.uint32)
    assert quiet.size == 2 * 64
    widened = (quiet << 16).astype(np.uint32).view(np.float32)
    np.testing.assert_array_equal(oracle.cast_bf16(widened), quiet.astype(np.uint16))


def test_signalling_nans_come_out_quiet():
    """IEEE 754-2019, 6.2: an operation on a signalling NaN delivers a quiet
    NaN.  Signalling fp32 NaNs of both signs (quiet bit clear, payload anywhere
    in the 22 bits below it) cast to quiet bf16 NaNs with the same sign."""
    rng = np.random.default_rng(3)
    payload = rng.integers(1, 1 << 22, size=20_000, dtype=np.uint32)
    sign = rng.integers(0, 2, size=payload.size, dtype=np.uint32) << 31
    snan = (sign | 0x7F800000 | payload).astype(np.uint32)
    out = oracle.cast_bf16(snan.view(np.float32))
    assert np.all((out & 0x7FC0) == 0x7FC0)                     # a quiet NaN
    np.testing.assert_array_equal(out >> 15, (snan >> 31).astype(np.uint16))
