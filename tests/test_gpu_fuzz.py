"""Seeded random cases of the main entry points against the oracle.

Each case draws a layout (tensor split, rank count, alignment, bucket), a
source count and dtype, an owner range and a flat sub-range inside it (starts
off the 8-element grid included), a source base, an output mode, non-zero
optimizer state and hyper-parameters, then checks every element in the range
bit for bit against the oracle and every element outside it unchanged.  The
8-bit-output updates and the clipped update are drawn the same way."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

SENTINEL_BF16 = 0x7E00          # a NaN pattern no update produces from finite inputs


def _layout(zb, rng):
    n_dp = int(rng.integers(1, 13))
    N = int(rng.integers(1, 120_000))
    k = int(rng.integers(1, 5))
    cuts = np.sort(rng.choice(np.arange(1, N), size=min(k - 1, N - 1), replace=False)) if N > 1 else []
    numels = np.diff(np.concatenate([[0], cuts, [N]])).astype(int).tolist()
    align = int(rng.choice([1, 2, 8, 64, 256]))
    bucket = int(rng.integers(1, 2 * N + 2))
    return zb.zero_layout(numels, n_dp, align=align, bucket_elems=bucket)


def _span(rng, lo, hi):
    """A non-empty [a, b) inside [lo, hi) (empty ranges are tested elsewhere)."""
    a, b = sorted(int(x) for x in rng.integers(lo, hi + 1, size=2))
    if a == b:
        a, b = (a - 1, a) if a > lo else (a, a + 1)
    return a, b


def _range(rng, L):
    rb = int(rng.integers(0, L.n_dp))
    re = int(rng.integers(rb + 1, L.n_dp + 1))
    a, b = _span(rng, rb * L.shard, re * L.shard)
    return rb, re, a, b


def _hp(rng):
    return oracle.AdamW(lr=float(rng.uniform(1e-5, 1e-2)), beta1=float(rng.uniform(0.5, 0.99)),
                        beta2=float(rng.uniform(0.9, 0.9999)), eps=float(10.0 ** rng.uniform(-10, -6)),
                        weight_decay=float(rng.uniform(0.0, 0.2)))


def _bf16_rows(rng, n_src, n, scale):
    x = torch.from_numpy((rng.standard_normal((n_src, n)) * scale).astype(np.float32))
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("case", range(40))
def test_fused_update(zlib, cuda_device, case):
    zb = zlib
    rng = np.random.default_rng(1000 + case)
    L = _layout(zb, rng)
    S, P = L.shard, L.padded_n
    rb, re, begin, end = _range(rng, L)
    n_src = int(rng.integers(1, 21))
    f32 = bool(rng.integers(0, 2))
    src_base = int(rng.integers(0, begin + 1))
    n_rows = end - src_base + int(rng.integers(0, 9))
    if f32:
        src = torch.from_numpy((rng.standard_normal((n_src, n_rows)) * 1e-2).astype(np.float32))
    else:
        src = _bf16_rows(rng, n_src, n_rows, 1e-2)
    own = (re - rb) * S
    w0 = (rng.standard_normal(own) * 0.02).astype(np.float32)
    m0 = (rng.standard_normal(own) * 1e-3).astype(np.float32)
    v0 = (rng.random(own) * 1e-6).astype(np.float32)
    shard_out = bool(rng.integers(0, 2))
    out_len = own if shard_out else P
    hp, t = _hp(rng), int(rng.integers(1, 1000))
    divisor = float(rng.choice([n_src, 3.0, 8.0, 0.5]))
    st = [torch.from_numpy(x.copy()).cuda() for x in (w0, m0, v0)]
    out = torch.full((out_len,), SENTINEL_BF16, dtype=torch.int16).view(torch.bfloat16).cuda()
    srcs = [src[r].cuda() for r in range(n_src)]
    zb.zero_reduce_scatter_adamw(L, srcs, zb.ZERO_F32 if f32 else zb.ZERO_BF16, src_base, divisor, rb, re,
                                 begin, end, *st, out, zb.ZERO_OUT_SHARD if shard_out else zb.ZERO_OUT_FULL,
                                 zb.ZeroAdamW.make(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, t))
    torch.cuda.synchronize()
    sel = slice(begin - rb * S, end - rb * S)
    rows = src[:, begin - src_base:end - src_base].contiguous()
    rows = rows.numpy() if f32 else parity.bits(rows)
    out_ref, *ref = oracle.rs_adamw_reference(rows, divisor, w0[sel], m0[sel], v0[sel], hp, t)
    what = f"case {case}: n_dp={L.n_dp} S={S} ranks {rb}..{re} [{begin}, {end}) n_src={n_src} f32={f32} "
    for got, init, r in zip(st, (w0, m0, v0), ref):
        g = parity.f32(got)
        parity.assert_bit_exact_f32(g[sel], r, what=what)
        outside = np.ones(own, bool)
        outside[sel] = False
        assert np.array_equal(g[outside].view(np.uint32), init[outside].view(np.uint32)), what + "outside"
    ob = parity.bits(out)
    osel = sel if shard_out else slice(begin, end)
    assert np.array_equal(ob[osel], out_ref), what + "bf16 output"
    rest = np.ones(out_len, bool)
    rest[osel] = False
    assert (ob[rest] == SENTINEL_BF16).all(), what + "output outside the range"


@pytest.mark.parametrize("case", range(20))
def test_accumulate(zlib, cuda_device, case):
    zb = zlib
    rng = np.random.default_rng(2000 + case)
    L = _layout(zb, rng)
    P = L.padded_n
    begin, end = _span(rng, 0, P)
    local = bool(rng.integers(0, 2))
    n_src = 1 if local else int(rng.integers(1, 17))
    src_base = int(rng.integers(0, begin + 1))
    dst_base = int(rng.integers(0, begin + 1))
    src = _bf16_rows(rng, n_src, end - src_base, 1e-2)
    d0 = (rng.standard_normal(end - dst_base) * 1e-2).astype(np.float32)
    first = bool(rng.integers(0, 2))
    dst = torch.from_numpy(d0.copy()).cuda()
    zb.zero_accumulate(L, zb.ZERO_ACC_LOCAL if local else zb.ZERO_ACC_REDUCE, [src[r].cuda() for r in range(n_src)],
                       zb.ZERO_BF16, src_base, dst, dst_base, begin, end, first)
    torch.cuda.synchronize()
    rows = parity.bits(src[:, begin - src_base:end - src_base].contiguous())
    acc = None if first else d0[begin - dst_base:end - dst_base]
    ref = oracle.accumulate_local(acc, rows[0], first) if local else oracle.accumulate_reduce(acc, rows, first)
    g = parity.f32(dst)
    what = f"case {case}: local={local} n_src={n_src} [{begin}, {end}) first={first} "
    parity.assert_bit_exact_f32(g[begin - dst_base:end - dst_base], ref, what=what)
    assert np.array_equal(g[:begin - dst_base].view(np.uint32), d0[:begin - dst_base].view(np.uint32)), what


@pytest.mark.parametrize("case", range(10))
def test_gather(zlib, cuda_device, case):
    zb = zlib
    rng = np.random.default_rng(3000 + case)
    L = _layout(zb, rng)
    S = L.shard
    shards = _bf16_rows(rng, L.n_dp, S, 1.0)
    full = torch.full((L.padded_n,), SENTINEL_BF16, dtype=torch.int16).view(torch.bfloat16).cuda()
    zb.zero_gather_layer(L, [shards[o].cuda() for o in range(L.n_dp)], full)
    torch.cuda.synchronize()
    assert np.array_equal(parity.bits(full), oracle.all_gather(parity.bits(shards))), f"case {case}"


@pytest.mark.parametrize("case", range(16))
def test_int8_gradient_paths(zlib, cuda_device, case):
    """8-bit gradients: each rank quantizes its gradient; then the update over a
    random owner sub-range and the accumulation over a random flat range."""
    zb = zlib
    rng = np.random.default_rng(4000 + case)
    L = _layout(zb, rng)
    S, P, n_dp = L.shard, L.padded_n, L.n_dp
    block = int(rng.choice([256, 512, 1024, 2048]))
    nb = -(-S // block)
    g = _bf16_rows(rng, n_dp, P, 1e-2)
    q = torch.empty((n_dp, P), dtype=torch.int8, device="cuda")
    sc = torch.empty((n_dp, max(n_dp * nb, 1)), device="cuda")
    for r in range(n_dp):
        zb.zero_quantize_int8(L, g[r].cuda(), q[r], sc[r], block)
    q_ref, s_ref = oracle.quantize_grad_int8(parity.bits(g), n_dp, block)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sc[:, :n_dp * nb].cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    deq = oracle.dequantize_grad_int8(q_ref, s_ref, n_dp, block)            # (n_dp, P) fp32
    qs, ss = [q[r] for r in range(n_dp)], [sc[r] for r in range(n_dp)]
    # the update over ranks rb..re-1, range [begin, end)
    rb, re, begin, end = _range(rng, L)
    own = (re - rb) * S
    w0 = (rng.standard_normal(own) * 0.02).astype(np.float32)
    m0 = (rng.standard_normal(own) * 1e-3).astype(np.float32)
    v0 = (rng.random(own) * 1e-6).astype(np.float32)
    st = [torch.from_numpy(x.copy()).cuda() for x in (w0, m0, v0)]
    out = torch.full((P,), SENTINEL_BF16, dtype=torch.int16).view(torch.bfloat16).cuda()
    hp, t = _hp(rng), int(rng.integers(1, 1000))
    zb.zero_reduce_scatter_adamw_int8(L, qs, ss, block, float(n_dp), rb, re, begin, end, *st, out,
                                      zb.ZERO_OUT_FULL,
                                      zb.ZeroAdamW.make(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, t))
    # the accumulation over [a, b) into a buffer based at a
    a, b = _span(rng, 0, P)
    A = torch.full((b - a,), 3.0, device="cuda")
    zb.zero_accumulate_int8(L, qs, ss, block, A, a, a, b, True)
    torch.cuda.synchronize()
    sel = slice(begin - rb * S, end - rb * S)
    out_ref, *ref = oracle.rs_adamw_reference(deq[:, begin:end].copy(), float(n_dp), w0[sel], m0[sel], v0[sel],
                                              hp, t)
    what = f"case {case}: n_dp={n_dp} S={S} block={block} ranks {rb}..{re} [{begin}, {end}) "
    for got, r in zip(st, ref):
        parity.assert_bit_exact_f32(parity.f32(got)[sel], r, what=what)
    ob = parity.bits(out)
    assert np.array_equal(ob[begin:end], out_ref), what + "bf16 output"
    rest = np.ones(P, bool)
    rest[begin:end] = False
    assert (ob[rest] == SENTINEL_BF16).all(), what + "output outside the range"
    A_ref = oracle.reduce_mean(deq[:, a:b].copy(), 1.0)
    parity.assert_bit_exact_f32(parity.f32(A)[:b - a], A_ref, what=f"case {case}: accumulation [{a}, {b}) ")


def _range256(rng, L):
    """Owners and a non-empty range on the 256-element grid (L laid out with align 256)."""
    rb = int(rng.integers(0, L.n_dp))
    re = int(rng.integers(rb + 1, L.n_dp + 1))
    blocks = (re - rb) * L.shard // 256
    a, b = _span(rng, 0, blocks)
    return rb, re, rb * L.shard + 256 * a, rb * L.shard + 256 * b


@pytest.mark.parametrize("case", range(12))
def test_updates_with_8bit_output(zlib, cuda_device, case):
    """The update writing the 8-bit block format, from bf16 gradients and from
    8-bit gradients: codes and scales equal the oracle's quantization of the
    oracle's bf16 result; the state as for the bf16 output."""
    zb = zlib
    rng = np.random.default_rng(5000 + case)
    n_dp = int(rng.integers(1, 13))
    L = zb.zero_layout([int(rng.integers(1, 120_000))], n_dp, align=256)
    S, P = L.shard, L.padded_n
    rb, re, begin, end = _range256(rng, L)
    own = (re - rb) * S
    sel = slice(begin - rb * S, end - rb * S)
    hp, t = _hp(rng), int(rng.integers(1, 1000))
    mk = lambda: zb.ZeroAdamW.make(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, t)
    w0 = (rng.standard_normal(own) * 0.02).astype(np.float32)
    m0 = (rng.standard_normal(own) * 1e-3).astype(np.float32)
    v0 = (rng.random(own) * 1e-6).astype(np.float32)
    g = _bf16_rows(rng, n_dp, P, 1e-2)
    block = int(rng.choice([256, 512, 1024, 2048]))
    nb = -(-S // block)
    q = torch.empty((n_dp, P), dtype=torch.int8, device="cuda")
    sc = torch.empty((n_dp, n_dp * nb), device="cuda")
    for r in range(n_dp):
        zb.zero_quantize_int8(L, g[r].cuda(), q[r], sc[r], block)
    q_ref, s_ref = oracle.quantize_grad_int8(parity.bits(g), n_dp, block)
    deq = oracle.dequantize_grad_int8(q_ref, s_ref, n_dp, block)
    for kind in ("bf16", "int8"):
        st = [torch.from_numpy(x.copy()).cuda() for x in (w0, m0, v0)]
        codes = torch.zeros(own, dtype=torch.int8, device="cuda")
        scales = torch.full((own // 256,), 9.0, device="cuda")
        if kind == "bf16":
            zb.zero_reduce_scatter_adamw_q8(L, [g[r].cuda() for r in range(n_dp)], zb.ZERO_BF16, 0, float(n_dp),
                                            rb, re, begin, end, *st, codes, scales, 256, mk())
            rows = parity.bits(g[:, begin:end].contiguous())
        else:
            zb.zero_reduce_scatter_adamw_int8_q8(L, [q[r] for r in range(n_dp)], [sc[r] for r in range(n_dp)],
                                                 block, float(n_dp), rb, re, begin, end, *st, codes, scales,
                                                 256, mk())
            rows = deq[:, begin:end].copy()
        torch.cuda.synchronize()
        out_ref, *ref = oracle.rs_adamw_reference(rows, float(n_dp), w0[sel], m0[sel], v0[sel], hp, t)
        what = f"case {case} {kind}: n_dp={n_dp} S={S} ranks {rb}..{re} [{begin}, {end}) "
        for got, r in zip(st, ref):
            parity.assert_bit_exact_f32(parity.f32(got)[sel], r, what=what)
        qo, so = oracle.quantize_int8(out_ref, 256)
        c = codes.cpu().numpy()
        assert np.array_equal(c[sel], qo), what + "codes"
        s8 = scales.cpu().numpy()
        k0 = (begin - rb * S) // 256
        assert np.array_equal(s8[k0:k0 + len(so)].view(np.uint32), so.view(np.uint32)), what + "scales"
        untouched = np.ones(own // 256, bool)
        untouched[k0:k0 + len(so)] = False
        assert (s8[untouched] == 9.0).all(), what + "scales outside the range"


@pytest.mark.parametrize("case", range(12))
def test_clipped_update(zlib, cuda_device, case):
    """The squared global norm over random buckets, then the clipped update:
    the norm within 1e-12 of the oracle's fp64 sum, the clip coefficient and so
    the state within the contract's tolerance (bit-exact whenever the fp32
    coefficient agrees)."""
    zb = zlib
    rng = np.random.default_rng(6000 + case)
    L = _layout(zb, rng)
    P, n_dp = L.padded_n, L.n_dp
    n_src = int(rng.integers(1, 13))
    g = _bf16_rows(rng, n_src, P, float(rng.choice([1e-3, 1.0, 30.0])))
    srcs = [g[r].cuda() for r in range(n_src)]
    divisor = float(n_src)
    max_norm = float(rng.choice([0.1, 1.0, 1e6]))
    bufs = zstep.NormBuffers("cuda")
    cuts = sorted({0, P, *(int(x) for x in rng.integers(0, P + 1, size=int(rng.integers(0, 4))))})
    for j, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        zb.zero_grad_norm_sq(L, srcs, zb.ZERO_BF16, 0, divisor, a, b, bufs.workspace, bufs.norm_sq, j > 0)
    torch.cuda.synchronize()
    rows = parity.bits(g)
    ref_norm = oracle.grad_norm_sq(rows, divisor)
    got_norm = float(bufs.norm_sq.item())
    assert abs(got_norm - ref_norm) <= 1e-12 * ref_norm + 1e-300, (case, got_norm, ref_norm)
    hp, t = _hp(rng), int(rng.integers(1, 1000))
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    z = np.zeros(P, np.float32)
    st = [torch.from_numpy(x.copy()).cuda() for x in (w0, z, z)]
    out = torch.empty(P, dtype=torch.bfloat16, device="cuda")
    zb.zero_reduce_scatter_adamw_clip(L, srcs, zb.ZERO_BF16, 0, divisor, 0, n_dp, 0, P, *st, out,
                                      zb.ZERO_OUT_FULL,
                                      zb.ZeroAdamW.make(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, t),
                                      bufs.norm_sq, max_norm)
    torch.cuda.synchronize()
    out_ref, *ref = oracle.rs_adamw_reference(rows, divisor, w0, z, z, hp, t, clip=(ref_norm, max_norm))
    parity.assert_state(st, ref, exact=False, what=f"case {case}: ")
    parity.assert_bf16_close(out, out_ref)
