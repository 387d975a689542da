"""CPU tests of the C ABI: the library builds and loads, exports every function
the header declares, its host-only calls agree with the oracle, and argument
checks reject bad calls before any CUDA call is made (no kernel runs here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from oracle import formulas
from zero_sharded_mixed_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zero_gb300.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(zero_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(zlib):
    names = _declared()
    assert {"zero_layout", "zero_reduce_scatter_adamw", "zero_gather_layer", "zero_accumulate",
            "zero_status_check", "zero_strerror"} <= set(names)
    lib = ctypes.CDLL(zlib.lib_path)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_layout_matches_oracle(zlib):
    rng = np.random.default_rng(0)
    for _ in range(3000):
        numels = rng.integers(0, 300, size=rng.integers(0, 5)).tolist()
        n_dp = int(rng.integers(1, 17))
        a = int(rng.choice([1, 2, 8, 64]))
        B = int(rng.integers(1, 2000))
        L, offs = zlib.zero_layout(numels, n_dp, align=a, bucket_elems=B, with_offsets=True)
        ref = oracle.layout(numels, n_dp, align=a, bucket=B)
        got = (L.n, L.shard, L.padded_n, L.bucket, L.n_buckets, L.n_dp, L.align)
        assert got == (ref["n"], ref["shard"], ref["padded"], ref["bucket"], ref["n_buckets"], n_dp, a)
        assert offs == ref["offsets"].tolist()


def test_workload_layouts_match_oracle(zlib):
    for numels, n_dp in [(inputs.gpt2xl_numels(), 8), (inputs.gpt2xl_numels(), 4),
                         (inputs.llama7b_numels(), 8), ([1 << 20], 4)]:
        L, offs = zlib.zero_layout(numels, n_dp, with_offsets=True)
        ref = oracle.layout(numels, n_dp)
        assert (L.n, L.shard, L.padded_n, L.n_buckets) == (ref["n"], ref["shard"], ref["padded"],
                                                          ref["n_buckets"])
        assert offs == ref["offsets"].tolist()
    for unit in inputs.llama7b_units():
        L = zlib.zero_layout(unit, 8)
        ref = oracle.layout(unit, 8)
        assert (L.shard, L.padded_n) == (ref["shard"], ref["padded"])


@pytest.mark.parametrize("args", [
    dict(n_dp=0), dict(align=0), dict(bucket_elems=0), dict(numels=[3, -1]),
])
def test_layout_errors(zlib, args):
    kw = dict(numels=[10], n_dp=2, align=8, bucket_elems=8)
    kw.update(args)
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_layout(kw.pop("numels"), **kw)
    assert e.value.code == zlib.ZERO_EINVAL
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_layout([2 ** 61, 2 ** 61], 2)
    assert e.value.code == zlib.ZERO_ERANGE


def test_bucket_and_shard_ranges(zlib):
    L = zlib.zero_layout([1000], 3, align=8, bucket_elems=100)
    assert (L.shard, L.padded_n, L.bucket, L.n_buckets) == (336, 1008, 104, 10)
    spans = [zlib.zero_bucket_range(L, b) for b in range(L.n_buckets)]
    assert spans[0] == (0, 104) and spans[-1] == (936, 1008)
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    assert [zlib.zero_shard_range(L, r) for r in range(3)] == [(0, 336, 336), (336, 672, 672),
                                                                (672, 1008, 1000)]
    for bad in (-1, L.n_buckets):
        with pytest.raises(zlib.ZeroError):
            zlib.zero_bucket_range(L, bad)
    with pytest.raises(zlib.ZeroError):
        zlib.zero_shard_range(L, 3)
    # a rank whose shard is all padding
    L = zlib.zero_layout([9], 4, align=8)
    assert zlib.zero_shard_range(L, 3) == (24, 32, 24)
    # a hand-made layout whose ranges would overflow int64 is refused
    L = zlib.zero_layout([1000], 3, align=8, bucket_elems=100)
    L.shard = 1 << 62
    with pytest.raises(zlib.ZeroError):
        zlib.zero_shard_range(L, 2)
    L = zlib.zero_layout([1000], 3, align=8, bucket_elems=100)
    L.bucket, L.n_buckets = 1 << 58, 8          # the library's element limit is 2^63 / 8
    with pytest.raises(zlib.ZeroError):
        zlib.zero_bucket_range(L, 4)
    assert zlib.zero_bucket_range(L, 0) == (0, L.padded_n)


def test_memory_and_comm_helpers_match_oracle(zlib):
    for N in (0, 1, 1000, 7e9, 7.5e9):
        for n in (1, 2, 8, 64):
            for s in range(4):
                assert zlib.zero_memory_bytes(N, n, s) == pytest.approx(formulas.zero_memory(N, n, s),
                                                                        rel=1e-12, abs=1e-9)
                assert zlib.zero_comm_bytes(N, n, s, 2, 4) == pytest.approx(
                    formulas.zero_comm_bytes(N, n, s, 2, 4), rel=1e-12, abs=1e-9)
    for bad in (-1, 4):
        with pytest.raises(zlib.ZeroError):
            zlib.zero_memory_bytes(10, 2, bad)
        with pytest.raises(zlib.ZeroError):
            zlib.zero_comm_bytes(10, 2, bad)


def test_strerror(zlib):
    assert zlib.zero_strerror(0) == "ok"
    for code in (-1, -2, -3, -4, -5):
        assert zlib.zero_strerror(code) and zlib.zero_strerror(code) != "unknown status code"
    assert zlib.zero_strerror(42) == "unknown status code"


# --------------------------------------------------------------------------
# argument checks that return before any CUDA call (fake, aligned pointers)
# --------------------------------------------------------------------------

FAKE = 0x10000   # never dereferenced: every case below fails a pure argument check


def _rs_call(zlib, **over):
    L = zlib.zero_layout([4096], 4)
    hp = zlib.ZeroAdamW.make(step=1)
    a = dict(L=ctypes.byref(L), src=None, n_src=4, dtype=zlib.ZERO_BF16, src_base=0, divisor=4.0,
             rb=0, re=4, begin=0, end=4096, w=FAKE, m=FAKE, v=FAKE, out=FAKE,
             mode=zlib.ZERO_OUT_FULL, hp=ctypes.byref(hp), stream=None)
    n_ptr = over.pop("n_ptrs", 4)
    ptrs = over.pop("ptrs", [FAKE] * n_ptr)
    a["src"] = (ctypes.c_void_p * max(1, len(ptrs)))(*ptrs)
    if "hp_fields" in over:
        for k, val in over.pop("hp_fields").items():
            setattr(hp, k, val)
    if "L_fields" in over:
        for k, val in over.pop("L_fields").items():
            setattr(L, k, val)
    a.update(over)
    return zlib.load().zero_reduce_scatter_adamw(
        a["L"], a["src"], a["n_src"], a["dtype"], a["src_base"], a["divisor"], a["rb"], a["re"],
        a["begin"], a["end"], a["w"], a["m"], a["v"], a["out"], a["mode"], a["hp"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(L=None), -1), (dict(hp=None), -1), (dict(w=None), -1), (dict(out=None), -1),
    (dict(n_src=0), -1), (dict(n_src=65, n_ptrs=65), -3), (dict(dtype=7), -1), (dict(mode=2), -1),
    (dict(rb=-1), -1), (dict(re=5), -1), (dict(rb=2, re=2), -1),
    (dict(rb=1, re=2, begin=0, end=1024), -1),        # range outside the owned shards
    (dict(begin=10, end=5), -1), (dict(end=4097), -1), (dict(src_base=8), -1),
    (dict(divisor=0.0), -1), (dict(divisor=float("inf")), -1), (dict(divisor=-1.0), -1),
    (dict(hp_fields=dict(step=0)), -1), (dict(hp_fields=dict(beta1=1.0)), -1),
    (dict(hp_fields=dict(lr=float("nan"))), -1),
    (dict(L_fields=dict(padded_n=4095)), -1),
    (dict(ptrs=[FAKE, FAKE, 0, FAKE]), -1),
    (dict(ptrs=[FAKE, FAKE + 1, FAKE, FAKE]), -2), (dict(w=FAKE + 2), -2), (dict(out=FAKE + 1), -2),
    (dict(begin=100, end=100), 0),                    # empty range: nothing to do
])
def test_rs_adamw_argument_checks(zlib, over, code):
    assert _rs_call(zlib, **over) == code


def test_internal_output_mode_is_refused(zlib):
    """out_mode -1 (the library's internal 8-bit-output marker) with a null
    output is refused by every public entry point with a bf16 output, even on
    an empty range, which returns before any launch; a mode outside {0, 1} or
    a null output with a valid mode is refused the same way."""
    lib = zlib.load()
    L = zlib.zero_layout([4096], 4)
    Lp = ctypes.byref(L)
    hp = zlib.ZeroAdamW.make(step=1)
    src = (ctypes.c_void_p * 4)(*[FAKE] * 4)
    norm = ctypes.c_void_p(FAKE)
    for mode, out in ((-1, None), (-1, FAKE), (2, FAKE), (0, None), (1, None)):
        assert _rs_call(zlib, mode=mode, out=out, begin=64, end=64) == -1, (mode, out)
        assert lib.zero_reduce_scatter_adamw_clip(Lp, src, 4, 0, 0, 4.0, 0, 4, 64, 64, FAKE, FAKE, FAKE,
                                                  out, mode, ctypes.byref(hp), norm, ctypes.c_float(1.0),
                                                  None) == -1, (mode, out)
        assert lib.zero_accumulate_adamw(Lp, 1, src, 1, 0, src, 4, 0, 4.0, 0, 4, 64, 64, FAKE, FAKE, FAKE,
                                         out, mode, ctypes.byref(hp), None) == -1, (mode, out)
        assert lib.zero_reduce_scatter_adamw_int8(Lp, src, src, 4, 256, 4.0, 0, 4, 64, 64, FAKE, FAKE, FAKE,
                                                  out, mode, ctypes.byref(hp), None) == -1, (mode, out)
    # the valid modes with an output still pass the empty-range call
    for mode in (0, 1):
        assert _rs_call(zlib, mode=mode, begin=64, end=64) == 0
        assert lib.zero_accumulate_adamw(Lp, 1, src, 1, 0, src, 4, 0, 4.0, 0, 4, 64, 64, FAKE, FAKE, FAKE,
                                         FAKE, mode, ctypes.byref(hp), None) == 0


def test_cast_argument_checks(zlib):
    """zero_cast_bf16 refuses a negative length, null pointers and misaligned
    pointers, and does nothing for n = 0, before any CUDA call."""
    lib = zlib.load()
    assert lib.zero_cast_bf16(FAKE, FAKE, -1, None) == -1
    assert lib.zero_cast_bf16(None, FAKE, 8, None) == -1
    assert lib.zero_cast_bf16(FAKE, None, 8, None) == -1
    assert lib.zero_cast_bf16(FAKE + 2, FAKE, 8, None) == -2
    assert lib.zero_cast_bf16(FAKE, FAKE + 1, 8, None) == -2
    assert lib.zero_cast_bf16(FAKE, FAKE, 0, None) == 0


def test_accumulate_and_gather_argument_checks(zlib):
    lib = zlib.load()
    L = zlib.zero_layout([4096], 4)
    src = (ctypes.c_void_p * 4)(*[FAKE] * 4)
    acc = lib.zero_accumulate
    Lp = ctypes.byref(L)
    assert acc(Lp, 9, src, 4, 0, 0, FAKE, 0, 0, 4096, 1, None) == -1        # mode
    assert acc(Lp, 0, src, 2, 0, 0, FAKE, 0, 0, 4096, 1, None) == -1        # LOCAL takes 1 source
    assert acc(Lp, 1, src, 0, 0, 0, FAKE, 0, 0, 4096, 1, None) == -1
    assert acc(Lp, 1, src, 65, 0, 0, FAKE, 0, 0, 4096, 1, None) == -3
    assert acc(Lp, 1, src, 4, 3, 0, FAKE, 0, 0, 4096, 1, None) == -1        # dtype
    assert acc(Lp, 1, src, 4, 0, 0, FAKE, 0, 0, 4097, 1, None) == -1        # past P
    assert acc(Lp, 1, src, 4, 0, 0, FAKE, 8, 0, 4096, 1, None) == -1        # dst_base > begin
    assert acc(Lp, 1, src, 4, 0, 0, FAKE + 2, 0, 0, 4096, 1, None) == -2    # dst alignment
    assert acc(Lp, 1, src, 4, 0, 0, None, 0, 0, 4096, 1, None) == -1
    assert acc(Lp, 1, src, 4, 0, 0, FAKE, 0, 64, 64, 1, None) == 0          # empty
    g = lib.zero_gather_layer
    assert g(None, src, FAKE, None) == -1
    assert g(Lp, src, None, None) == -1
    bad = (ctypes.c_void_p * 4)(FAKE, 0, FAKE, FAKE)
    assert g(Lp, bad, FAKE, None) == -1
    odd = (ctypes.c_void_p * 4)(FAKE, FAKE + 1, FAKE, FAKE)
    assert g(Lp, odd, FAKE, None) == -2
    empty = zlib.zero_layout([0], 4)
    assert g(ctypes.byref(empty), src, FAKE, None) == 0


def test_int8_gradient_argument_checks(zlib):
    """zero_reduce_scatter_adamw_int8 and zero_accumulate_int8 refuse bad
    arguments before touching any pointer."""
    lib = zlib.load()
    L = zlib.zero_layout([4096], 4)
    Lp = ctypes.byref(L)
    q = (ctypes.c_void_p * 4)(*[FAKE] * 4)
    s = (ctypes.c_void_p * 4)(*[FAKE] * 4)
    hp = zlib.ZeroAdamW.make(step=1)
    hpp = ctypes.byref(hp)

    def rs(q=q, s=s, n=4, block=256, div=4.0, rb=0, re=4, b=0, e=4096, w=FAKE, mode=0, h=hpp):
        return lib.zero_reduce_scatter_adamw_int8(Lp, q, s, n, block, div, rb, re, b, e,
                                                  w, FAKE, FAKE, FAKE, mode, h, None)

    assert rs(q=None) == -1
    assert rs(n=0) == -1
    assert rs(n=65) == -3
    for block in (0, 128, 384, 4096):
        assert rs(block=block) == -1
    assert rs(s=(ctypes.c_void_p * 4)(FAKE, FAKE + 2, FAKE, FAKE)) == -2     # scales 4-byte aligned
    assert rs(q=(ctypes.c_void_p * 4)(FAKE, 0, FAKE, FAKE)) == -1
    assert rs(div=0.0) == -1
    assert rs(rb=1, b=0) == -1                                               # begin below the owners
    assert rs(e=4097) == -1
    assert rs(mode=7) == -1
    assert rs(w=FAKE + 2) == -2
    assert rs(h=None) == -1
    assert rs(b=64, e=64) == 0                                               # empty
    acc = lib.zero_accumulate_int8
    assert acc(None, q, s, 4, 256, FAKE, 0, 0, 4096, 1, None) == -1
    assert acc(Lp, q, s, 4, 256, None, 0, 0, 4096, 1, None) == -1
    assert acc(Lp, q, s, 4, 100, FAKE, 0, 0, 4096, 1, None) == -1           # block
    assert acc(Lp, q, s, 65, 256, FAKE, 0, 0, 4096, 1, None) == -3
    assert acc(Lp, q, s, 4, 256, FAKE, 8, 0, 4096, 1, None) == -1           # dst_base > begin
    assert acc(Lp, q, s, 4, 256, FAKE, 0, 0, 4097, 1, None) == -1           # past P
    assert acc(Lp, q, s, 4, 256, FAKE + 2, 0, 0, 4096, 1, None) == -2       # dst alignment
    assert acc(Lp, q, s, 4, 256, FAKE, 0, 64, 64, 1, None) == 0             # empty


def test_q8_update_argument_checks(zlib):
    """zero_reduce_scatter_adamw_q8 refuses a block other than 256 and ranges or
    shards off the 256-element grid before touching any pointer."""
    lib = zlib.load()
    L = zlib.zero_layout([4096], 4, align=256)
    L8 = zlib.zero_layout([4000], 4, align=8)                # S = 1000: off the grid
    src = (ctypes.c_void_p * 4)(*[FAKE] * 4)
    hp = zlib.ZeroAdamW.make(step=1)

    def q8(Lx=L, block=256, b=0, e=4096, q=FAKE, sc=FAKE, dt=0):
        return lib.zero_reduce_scatter_adamw_q8(ctypes.byref(Lx), src, 4, dt, 0, 4.0, 0, 4, b, e,
                                                FAKE, FAKE, FAKE, q, sc, block, ctypes.byref(hp), None)

    assert q8(block=512) == -1
    assert q8(Lx=L8, e=4000) == -1
    assert q8(b=8) == -1 and q8(e=4088) == -1
    assert q8(q=None) == -1 and q8(sc=None) == -1
    assert q8(sc=FAKE + 2) == -2
    assert q8(dt=5) == -1
    assert q8(b=512, e=512) == 0                                # empty
    s8 = (ctypes.c_void_p * 4)(*[FAKE] * 4)

    def iq8(Lx=L, out_block=256, b=0, e=4096, q=FAKE, block=256):
        return lib.zero_reduce_scatter_adamw_int8_q8(ctypes.byref(Lx), src, s8, 4, block, 4.0, 0, 4, b, e,
                                                     FAKE, FAKE, FAKE, q, FAKE, out_block,
                                                     ctypes.byref(hp), None)

    assert iq8(out_block=512) == -1 and iq8(block=100) == -1
    assert iq8(Lx=L8, e=4000) == -1 and iq8(b=8) == -1
    assert iq8(q=None) == -1
    assert iq8(b=256, e=256) == 0


def test_missing_library_fails_loudly(zlib, monkeypatch, tmp_path):
    from zero_sharded_mixed_gb300 import binding
    monkeypatch.setattr(binding, "lib_path", str(tmp_path / "nope.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(ImportError):
        binding.load()


def test_schedule_fill_matches_the_oracle_bias_corrections(zlib):
    """The device-schedule table holds exactly the by-value scalars: lr and the
    oracle's bias corrections of every step."""
    import oracle
    hp = zlib.ZeroAdamW.make(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    table = zlib.zero_schedule_fill(hp, 5, 20)
    o = oracle.AdamW(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    for k in range(20):
        bc1, bc2 = oracle.bias_corrections(o, 5 + k)
        assert table[k].tolist() == [float(np.float32(3e-4)), float(bc1), float(bc2)]
    lrs = [1e-3 * (k + 1) for k in range(4)]
    t2 = zlib.zero_schedule_fill(hp, 1, 4, lrs)
    assert t2[:, 0].tolist() == [float(np.float32(x)) for x in lrs]
    lib = zlib.load()
    assert lib.zero_schedule_fill(None, 1, 4, None, FAKE) == -1
    assert lib.zero_schedule_fill(ctypes.byref(hp), 0, 4, None, FAKE) == -1
    assert lib.zero_schedule_fill(ctypes.byref(hp), 1, 0, None, FAKE) == -1
    assert lib.zero_schedule_fill(ctypes.byref(hp), (1 << 63) - 1, 2, None, FAKE) == -1   # step past int64
    assert lib.zero_schedule_fill(ctypes.byref(hp), 1, 1 << 62, None, FAKE) == -1         # index past int64
    assert lib.zero_schedule_advance(None, 4, FAKE, FAKE, None) == -1
    assert lib.zero_schedule_advance(FAKE, 0, FAKE, FAKE, None) == -1
    assert lib.zero_schedule_advance(FAKE, 4, FAKE + 4, FAKE, None) == -2      # index 8-byte aligned


def test_layout_whose_size_overflows_is_refused(zlib):
    """A hand-made layout whose shard * n_dp overflows int64 (2^62 * 4 wraps to
    0, the padded_n given) is refused by every entry point that takes a
    layout, even on an empty range, which returns before any launch; the
    same calls with zero_layout's own layout pass."""
    lib = zlib.load()
    good = zlib.zero_layout([4096], 4)
    bad = zlib.zero_layout([4096], 4)
    bad.shard, bad.padded_n, bad.n = 1 << 62, 0, 0
    src = (ctypes.c_void_p * 4)(*[FAKE] * 4)
    hp = zlib.ZeroAdamW.make(step=1)
    hpp = ctypes.byref(hp)
    for L, want in ((good, 0), (bad, -1)):
        Lp = ctypes.byref(L)
        assert lib.zero_reduce_scatter_adamw(Lp, src, 4, 0, 0, 4.0, 0, 4, 0, 0, FAKE, FAKE, FAKE, FAKE, 0,
                                             hpp, None) == want
        assert lib.zero_reduce_scatter_adamw_int8(Lp, src, src, 4, 256, 4.0, 0, 4, 0, 0, FAKE, FAKE, FAKE,
                                                  FAKE, 0, hpp, None) == want
        assert lib.zero_accumulate(Lp, 1, src, 4, 0, 0, FAKE, 0, 0, 0, 1, None) == want
        assert lib.zero_accumulate_int8(Lp, src, src, 4, 256, FAKE, 0, 0, 0, 1, None) == want
        assert lib.zero_accumulate_adamw(Lp, 1, src, 1, 0, src, 4, 0, 4.0, 0, 4, 0, 0, FAKE, FAKE, FAKE,
                                         FAKE, 0, hpp, None) == want
    Lp = ctypes.byref(bad)
    assert lib.zero_gather_layer(Lp, src, FAKE, None) == -1
    assert lib.zero_quantize_int8(Lp, FAKE, FAKE, FAKE, 256, None) == -1
    assert lib.zero_gather_layer_int8(Lp, src, src, 256, FAKE, None) == -1
    assert lib.zero_grad_norm_sq(Lp, src, 4, 0, 0, 4.0, 0, 0, FAKE, 1 << 20, FAKE, 0, None) == -1
