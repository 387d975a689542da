"""zero_cast_bf16 (the library's fp32 -> bf16 cast of weights) against the
oracle's round-to-nearest-even cast, bit for bit, through the C ABI.

"ZeRO and FSDP", "The idea, one stage at a time": the owners cast their fp32
master shards to bf16 before the all-gather.  Inputs: every bit-pattern class
(random 32-bit patterns, so NaNs with payloads of both signs, infinities,
subnormals and zeros appear), exact ties either side of even, values that
round up to infinity, lengths that leave a ragged tail or none, and a source
off the 16-byte grid (the scalar path).  Elements past n are left alone.  The
engines' first bf16 weights are the same cast of their master weights."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

SENTINEL = 0x7E5A     # a bf16 pattern the cast never writes for the inputs below past n


def _dev_f32(bits_u32):
    return torch.from_numpy(np.ascontiguousarray(bits_u32, dtype=np.uint32).view(np.float32).copy()).cuda()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _special_patterns():
    vals = [
        0x00000000, 0x80000000,                          # +-0
        0x00000001, 0x807fffff, 0x00008000, 0x00018000,   # subnormals, incl. ties
        0x3f808000, 0x3f818000, 0xbf808000, 0xbf818000,   # exact ties: stay even / go up to even
        0x3f808001, 0x3f807fff,                           # just above / below a tie
        0x7f7f7fff, 0x7f7f8000, 0x7f7fffff,               # largest finite: stays / tie to inf / rounds to inf
        0xff7f8000, 0xff7fffff,
        0x7f800000, 0xff800000,                           # +-inf
        0x7fc00000, 0xffc00000, 0x7f800001, 0xff800001,   # quiet and signalling NaNs
        0x7fa5a5a5, 0xffbfffff, 0x7fffffff, 0x7f80ffff,   # NaN payloads, incl. only low payload bits
    ]
    return np.array(vals, dtype=np.uint32)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 27, 4096, 1_000_003, 4_194_304])
def test_cast_matches_oracle_bit_for_bit(zlib, cuda_device, n):
    rng = np.random.default_rng(n)
    bits = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    sp = _special_patterns()
    bits[:min(n, sp.size)] = sp[:min(n, sp.size)]
    src = _dev_f32(bits)
    dst = torch.full((n + 16,), int(np.uint16(SENTINEL).view(np.int16)), dtype=torch.int16, device="cuda")
    zlib.zero_cast_bf16(src, dst.view(torch.bfloat16), n)
    torch.cuda.synchronize()
    got = _bits(dst)
    ref = oracle.cast_bf16(bits.view(np.float32))
    assert np.array_equal(got[:n], ref), int((got[:n] != ref).sum())
    assert (got[n:] == SENTINEL).all()


def test_cast_specials_by_value(zlib, cuda_device):
    """The special cases by their expected bf16 patterns, written out."""
    sp = _special_patterns()
    src = _dev_f32(sp)
    dst = torch.empty(sp.size, dtype=torch.bfloat16, device="cuda")
    zlib.zero_cast_bf16(src, dst)
    torch.cuda.synchronize()
    got = dict(zip(sp.tolist(), _bits(dst).tolist()))
    assert got[0x3f808000] == 0x3f80 and got[0x3f818000] == 0x3f82       # ties to even
    assert got[0xbf808000] == 0xbf80 and got[0xbf818000] == 0xbf82
    assert got[0x3f808001] == 0x3f81 and got[0x3f807fff] == 0x3f80
    assert got[0x7f7f7fff] == 0x7f7f and got[0x7f7f8000] == 0x7f80        # tie at the top goes to inf
    assert got[0x7f7fffff] == 0x7f80 and got[0xff7fffff] == 0xff80
    assert got[0x7f800000] == 0x7f80 and got[0xff800000] == 0xff80
    assert got[0x00000001] == 0x0000 and got[0x00018000] == 0x0002        # subnormal tie to even
    assert got[0x80000000] == 0x8000
    assert got[0x7f800001] == 0x7fc0 and got[0xff800001] == 0xffc0        # signalling NaN made quiet
    assert got[0x7fa5a5a5] == 0x7fe5 and got[0xffbfffff] == 0xffff       # payload kept, quiet bit set
    assert got[0x7f80ffff] == 0x7fc0                                      # low payload only: still a NaN


def test_cast_off_the_vector_grid(zlib, cuda_device):
    """A source and destination one element past a 16-byte boundary take the
    scalar path; the result is the same."""
    n = 100_003
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 32, size=n + 1, dtype=np.uint64).astype(np.uint32)
    src = _dev_f32(bits)
    dst = torch.zeros(n + 2, dtype=torch.bfloat16, device="cuda")
    zlib.zero_cast_bf16(src[1:], dst[1:], n)
    torch.cuda.synchronize()
    got = _bits(dst)
    assert np.array_equal(got[1:n + 1], oracle.cast_bf16(bits[1:].view(np.float32)))
    assert got[0] == 0 and got[n + 1] == 0


def test_cast_argument_checks(zlib, cuda_device):
    src = torch.zeros(16, device="cuda")
    dst = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    zlib.zero_cast_bf16(src, dst, 0)                       # nothing to do
    lib = zlib.load()
    assert lib.zero_cast_bf16(src.data_ptr(), dst.data_ptr(), -1, None) == zlib.ZERO_EINVAL
    assert lib.zero_cast_bf16(None, dst.data_ptr(), 4, None) == zlib.ZERO_EINVAL
    assert lib.zero_cast_bf16(src.data_ptr() + 2, dst.data_ptr(), 4, None) == zlib.ZERO_EALIGN
    assert lib.zero_cast_bf16(src.data_ptr(), dst.data_ptr() + 1, 4, None) == zlib.ZERO_EALIGN
    host = torch.zeros(16)
    assert lib.zero_cast_bf16(host.data_ptr(), dst.data_ptr(), 4, None) == zlib.ZERO_EINVAL
    with pytest.raises(ValueError):
        zlib.zero_cast_bf16(src, dst, 17)


def test_engines_start_from_the_cast_master_weights(zlib, cuda_device):
    """The first bf16 weights of both engines are the oracle's cast of their
    master weights."""
    from zero_sharded_mixed_gb300 import ZeroConfig, Zero3Engine, ZeroEngine
    from zero_sharded_mixed_gb300 import inputs
    N = 10_007
    w = inputs.master_weights(N, N, seed=3)
    cfg = ZeroConfig.from_dict({"zero_optimization": {"stage": 2}})
    L = zlib.zero_layout([N], 4)
    master = torch.zeros(L.padded_n, device="cuda")
    master[:N] = w.cuda()
    eng = ZeroEngine([N], 4, cfg, master=master)
    ref = oracle.cast_bf16(master.cpu().numpy())
    assert np.array_equal(_bits(eng.out), ref)
    cfg3 = ZeroConfig.from_dict({"zero_optimization": {"stage": 3}})
    units = [[N], [513, 7]]
    masters = []
    for u in units:
        Lu = zlib.zero_layout(u, 4)
        x = torch.zeros(Lu.padded_n, device="cuda")
        x[:Lu.n] = inputs.master_weights(Lu.n, Lu.n, seed=len(masters) + 7).cuda()
        masters.append(x)
    eng3 = Zero3Engine(units, 4, cfg3, masters=masters)
    for u, x in zip(eng3.units, masters):
        assert np.array_equal(_bits(u.shards.reshape(-1)), oracle.cast_bf16(x.cpu().numpy()))
