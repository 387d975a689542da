"""Parity of the fused reduce-scatter + AdamW + cast + gather kernel against the
oracle, element by element, through the C ABI (zero_reduce_scatter_adamw)."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

HP_ORACLE = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


def _hp(zb, t, hp=HP_ORACLE):
    return zb.ZeroAdamW.make(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, t)


def _setup(zb, N, n_dp, align=8, bucket=500_000_000, seed=0, device="cuda"):
    L = zb.zero_layout([N], n_dp, align=align, bucket_elems=bucket)
    P = L.padded_n
    w = inputs.master_weights(N, P, seed=seed)
    state = [w.to(device), torch.zeros(P, device=device), torch.zeros(P, device=device)]
    out = torch.zeros(P, dtype=torch.bfloat16, device=device)
    return L, state, out


def _grads_cpu(L, seed, step, **kw):
    return inputs.grads_bf16(L.n_dp, L.n, L.padded_n, seed=seed, step=step, **kw)


def _oracle_full_step(g_cpu, state_np, n_dp, t, hp=HP_ORACLE):
    w, m, v = state_np
    S = w.size // n_dp
    full, w2, m2, v2 = oracle.zero_step(parity.bits(g_cpu), w.reshape(n_dp, S), m.reshape(n_dp, S),
                                        v.reshape(n_dp, S), hp, t)
    return full[0], [w2.reshape(-1), m2.reshape(-1), v2.reshape(-1)]


def test_tiny_zero1_three_steps(zlib, cuda_device):
    """N = 2^20 fp32 params ~ N(0, 0.02), n_dp = 4 ranks with bf16 grads
    ~ N(0, 1e-3), m = v = 0, AdamW lr 1e-4 (0.9, 0.999) eps 1e-8 wd 0.1,
    3 steps, seed 0."""
    zb = zlib
    L, state, out = _setup(zb, 1 << 20, 4)
    ref = [parity.f32(x) for x in state]
    for t in (1, 2, 3):
        g = _grads_cpu(L, 0, t)
        gd = [g[r].to("cuda") for r in range(L.n_dp)]
        zstep.zero12_step(L, gd, *state, out, _hp(zb, t))
        torch.cuda.synchronize()
        ref_out, ref = _oracle_full_step(g, ref, L.n_dp, t)
        parity.assert_state(state, ref, what=f"t={t} ")
        parity.assert_bf16_close(out, ref_out)
        assert np.array_equal(parity.bits(out), ref_out)


@pytest.mark.parametrize("N,n_dp,bucket", [(100_003, 3, 30_000), (65_541, 8, 500_000_000)])
def test_sharded_step_equals_data_parallel(zlib, cuda_device, N, n_dp, bucket):
    """"ZeRO and FSDP", "The idea, one stage at a time": ZeRO-1/2 computes the
    same step as plain data parallelism.  The library's sharded step (each
    owner updates its shard, the bf16 result gathered into the full buffer)
    against the oracle's data-parallel step (an all-reduce mean, then AdamW on
    the full vector by every rank): the concatenated fp32 state equals every
    rank's full copy, and the gathered bf16 weights every rank's, bit for bit,
    over three steps."""
    zb = zlib
    L, state, out = _setup(zb, N, n_dp, bucket=bucket, seed=7)
    P = L.padded_n
    w0 = parity.f32(state[0])
    full_w = np.tile(w0, (n_dp, 1))
    full_m = np.zeros((n_dp, P), np.float32)
    full_v = np.zeros((n_dp, P), np.float32)
    for t in (1, 2, 3):
        g = _grads_cpu(L, 7, t)
        zstep.zero12_step(L, [g[r].to("cuda") for r in range(n_dp)], *state, out, _hp(zb, t))
        torch.cuda.synchronize()
        dp_out, full_w, full_m, full_v = oracle.dp_step(parity.bits(g), full_w, full_m, full_v, HP_ORACLE, t)
        for r in range(n_dp):
            for got, ref in zip(state, (full_w[r], full_m[r], full_v[r])):
                parity.assert_bit_exact_f32(got, ref, what=f"t={t} rank {r} ")
            assert np.array_equal(parity.bits(out), dp_out[r]), f"t={t} rank {r} bf16"


@pytest.mark.parametrize("n_dp", [1, 2, 3, 4, 5, 7, 8, 16])
@pytest.mark.parametrize("align", [8, 1])
def test_ragged_sizes_and_rank_counts(zlib, cuda_device, n_dp, align):
    zb = zlib
    N = 40_000 + 13 * n_dp + 5          # several CTAs' worth and a ragged tail
    L, state, out = _setup(zb, N, n_dp, align=align, bucket=7_777, seed=n_dp)
    ref = [parity.f32(x) for x in state]
    for t in (1, 2):
        g = _grads_cpu(L, n_dp, t)
        gd = [g[r].to("cuda") for r in range(n_dp)]
        zstep.zero12_step(L, gd, *state, out, _hp(zb, t))
        torch.cuda.synchronize()
        ref_out, ref = _oracle_full_step(g, ref, n_dp, t)
        parity.assert_state(state, ref, what=f"n_dp={n_dp} a={align} t={t} ")
        assert np.array_equal(parity.bits(out), ref_out)
    # the padding stays exactly zero
    assert not parity.f32(state[0])[N:].any() and not parity.bits(out)[N:].any()


@pytest.mark.parametrize("bucket", [8, 1000, 4096, 12_345, 10 ** 9])
def test_bucketing_is_invisible(zlib, cuda_device, bucket):
    zb = zlib
    N, n_dp = 50_000, 4
    L, state, out = _setup(zb, N, n_dp, bucket=bucket)
    Lref, sref, oref = _setup(zb, N, n_dp, bucket=10 ** 9)
    g = _grads_cpu(L, 3, 1)
    gd = [g[r].to("cuda") for r in range(n_dp)]
    zstep.zero12_step(L, gd, *state, out, _hp(zb, 1))
    zstep.zero12_step(Lref, gd, *sref, oref, _hp(zb, 1))
    torch.cuda.synchronize()
    for a, b in zip(state, sref):
        parity.assert_bit_exact_f32(a, b)
    assert torch.equal(out.view(torch.int16), oref.view(torch.int16))


def test_one_owned_shard_writes_only_its_part(zlib, cuda_device):
    """The 7B-shaped configuration in small: one owner, its n_dp gradient slices,
    bf16 written into the full buffer at its offset; the rest untouched."""
    zb = zlib
    N, n_dp, o = 100_003, 8, 5
    L = zb.zero_layout([N], n_dp)
    S, P = L.shard, L.padded_n
    g = inputs.grads_bf16(n_dp, N, P, seed=9, step=1, outlier_p=0.01)
    slices = [g[r, o * S:(o + 1) * S].contiguous().cuda() for r in range(n_dp)]
    w0 = inputs.master_weights(N, P, seed=9)[o * S:(o + 1) * S].contiguous()
    st = [w0.cuda(), torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")]
    canary = torch.full((P,), 12345, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    out = canary.clone()
    zstep.zero12_step(L, slices, *st, out, _hp(zb, 1), rank_begin=o, rank_end=o + 1,
                      grad_base=o * S)
    torch.cuda.synchronize()
    src = parity.bits(torch.stack([s.cpu() for s in slices]))
    ref_out, w, m, v = oracle.rs_adamw_reference(src, n_dp, parity.f32(w0), np.zeros(S, np.float32),
                                                 np.zeros(S, np.float32), HP_ORACLE, 1)
    parity.assert_state(st, [w, m, v])
    ob = parity.bits(out)
    assert np.array_equal(ob[o * S:(o + 1) * S], ref_out)
    assert np.all(ob[: o * S] == 12345) and np.all(ob[(o + 1) * S:] == 12345)


def test_out_shard_mode_and_fp32_sources(zlib, cuda_device):
    zb = zlib
    N, n_dp = 33_031, 3
    L = zb.zero_layout([N], n_dp)
    S, P = L.shard, L.padded_n
    rng = np.random.default_rng(5)
    acc = (rng.standard_normal((n_dp, P)) * 1e-3).astype(np.float32)
    acc[:, N:] = 0
    w0 = parity.f32(inputs.master_weights(N, P, seed=5))
    st = [torch.from_numpy(w0.copy()).cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    own = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    srcs = [torch.from_numpy(acc[r].copy()).cuda() for r in range(n_dp)]
    divisor = float(n_dp * 4)
    zb.zero_reduce_scatter_adamw(L, srcs, zb.ZERO_F32, 0, divisor, 0, n_dp, 0, P, *st, own,
                                 zb.ZERO_OUT_SHARD, _hp(zb, 7))
    torch.cuda.synchronize()
    ref_out, w, m, v = oracle.rs_adamw_reference(acc, divisor, w0, np.zeros(P, np.float32),
                                                 np.zeros(P, np.float32), HP_ORACLE, 7)
    parity.assert_state(st, [w, m, v])
    assert np.array_equal(parity.bits(own), ref_out)


@pytest.mark.parametrize("n", [1, 2, 7, 8, 9, 15, 17, 255, 256 * 8 + 3])
def test_short_and_misaligned_ranges(zlib, cuda_device, n):
    """Ragged lengths take the vector body plus a scalar tail; a range that
    starts off a 16-byte boundary takes the element-wise kernel."""
    zb = zlib
    n_dp = 2
    for start in (0, 1, 3):
        N = start + n
        L = zb.zero_layout([N], 1, align=1)     # one owner holding everything
        g = inputs.grads_bf16(n_dp, N, N, seed=n, step=1)
        w0 = inputs.master_weights(N, N, seed=n)
        st = [w0.cuda(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
        out = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
        gd = [g[r].cuda() for r in range(n_dp)]
        zb.zero_reduce_scatter_adamw(L, gd, zb.ZERO_BF16, 0, float(n_dp), 0, 1, start, N,
                                     *st, out, zb.ZERO_OUT_FULL, _hp(zb, 2))
        torch.cuda.synchronize()
        ref_out, w, m, v = oracle.rs_adamw_reference(parity.bits(g)[:, start:], n_dp,
                                                     parity.f32(w0)[start:], np.zeros(n, np.float32),
                                                     np.zeros(n, np.float32), HP_ORACLE, 2)
        parity.assert_state([x[start:] for x in st], [w, m, v], what=f"start={start} ")
        assert np.array_equal(parity.bits(out)[start:], ref_out)
        # elements before the range are untouched
        assert np.array_equal(parity.f32(st[0])[:start], parity.f32(w0)[:start])
        assert not parity.bits(out)[:start].any()


def test_special_values_propagate(zlib, cuda_device):
    zb = zlib
    n_dp, N = 2, 64
    L = zb.zero_layout([N], 1)
    gf = np.zeros((n_dp, N), np.float32)
    gf[0, :8] = [np.nan, np.inf, -np.inf, 0.0, -0.0, 1e38, -1e38, 3e-39]
    gf[1, :8] = [1.0, 1.0, 1.0, -0.0, -0.0, 1e38, -1e38, 3e-39]
    gf[:, 8:] = np.linspace(-1, 1, N - 8, dtype=np.float32)
    g = oracle.cast_bf16(gf)
    w0 = np.linspace(-0.05, 0.05, N, dtype=np.float32)
    w0[16] = 3.3e38                    # a weight near the top of the bf16 range
    st = [torch.from_numpy(w0.copy()).cuda(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
    out = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    gd = [inputs.from_bf16_bits(g[r], "cuda") for r in range(n_dp)]
    zb.zero_reduce_scatter_adamw(L, gd, zb.ZERO_BF16, 0, float(n_dp), 0, 1, 0, N, *st, out,
                                 zb.ZERO_OUT_FULL, _hp(zb, 1))
    torch.cuda.synchronize()
    ref_out, w, m, v = oracle.rs_adamw_reference(g, n_dp, w0, np.zeros(N, np.float32),
                                                 np.zeros(N, np.float32), HP_ORACLE, 1)
    parity.assert_state(st, [w, m, v])
    parity.assert_bf16_close(out, ref_out, ulps=0)


def test_zero_length_range_is_a_no_op(zlib, cuda_device):
    zb = zlib
    L = zb.zero_layout([64], 2)
    g = [torch.zeros(64, dtype=torch.bfloat16, device="cuda")] * 2
    st = [torch.ones(64, device="cuda") for _ in range(3)]
    out = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    zb.zero_reduce_scatter_adamw(L, g, zb.ZERO_BF16, 0, 2.0, 0, 2, 10, 10, *st, out,
                                 zb.ZERO_OUT_FULL, _hp(zb, 1))
    zb.zero_status_check()
    assert all(torch.all(x == 1) for x in st) and not out.view(torch.int16).any()


@pytest.mark.parametrize("n_src,dtype", [(1, "bf16"), (2, "bf16"), (1, "f32"), (2, "f32"), (8, "bf16")])
def test_several_waves_with_partial_groups(zlib, cuda_device, n_src, dtype):
    """5,000,011 elements: several grid-stride passes of the multi-vector loop,
    a partial last group and a ragged tail."""
    zb = zlib
    N = 5_000_011
    L = zb.zero_layout([N], 1, align=1)
    rng = np.random.default_rng(n_src)
    xf = (rng.standard_normal((n_src, N)) * 1e-3).astype(np.float32)
    if dtype == "bf16":
        src_np = oracle.cast_bf16(xf)
        srcs = [inputs.from_bf16_bits(src_np[r], "cuda") for r in range(n_src)]
        code = zb.ZERO_BF16
    else:
        src_np = xf
        srcs = [torch.from_numpy(xf[r].copy()).cuda() for r in range(n_src)]
        code = zb.ZERO_F32
    w0 = parity.f32(inputs.master_weights(N, N, seed=n_src))
    m0 = (np.abs(rng.standard_normal(N)) * 1e-4).astype(np.float32)
    v0 = (np.abs(rng.standard_normal(N)) * 1e-8).astype(np.float32)
    st = [torch.from_numpy(x.copy()).cuda() for x in (w0, m0, v0)]
    out = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    zb.zero_reduce_scatter_adamw(L, srcs, code, 0, float(n_src), 0, 1, 0, N, *st, out,
                                 zb.ZERO_OUT_FULL, _hp(zb, 4))
    torch.cuda.synchronize()
    ref_out, w, m, v = oracle.rs_adamw_reference(src_np, n_src, w0, m0, v0, HP_ORACLE, 4)
    parity.assert_state(st, [w, m, v])
    assert np.array_equal(parity.bits(out), ref_out)


@pytest.mark.parametrize("n_src,dtype", [(6, "bf16"), (32, "bf16"), (64, "bf16"), (3, "f32"),
                                         (64, "f32")])
def test_source_counts_up_to_the_limit(zlib, cuda_device, n_src, dtype):
    """Every source count the kernels take, up to ZERO_MAX_SRC = 64: the
    compile-time counts and the runtime-count kernel, bf16 and fp32 sources,
    a ragged tail; two steps against the oracle, bit for bit."""
    zb = zlib
    assert zb.ZERO_MAX_SRC == 64
    N = 1000 * n_src + 7
    L = zb.zero_layout([N], n_src)
    P = L.padded_n
    w0 = inputs.master_weights(N, P, seed=n_src)
    st = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    ref = [parity.f32(w0), np.zeros(P, np.float32), np.zeros(P, np.float32)]
    for t in (1, 2):
        g = inputs.grads_bf16(n_src, N, P, seed=n_src, step=t)
        if dtype == "bf16":
            srcs, dt, rows = [g[r].cuda() for r in range(n_src)], zb.ZERO_BF16, parity.bits(g)
        else:
            gf = (g.float() * 3.0).contiguous()            # fp32 sources not on the bf16 grid
            srcs, dt, rows = [gf[r].cuda() for r in range(n_src)], zb.ZERO_F32, gf.numpy()
        zb.zero_reduce_scatter_adamw(L, srcs, dt, 0, float(n_src), 0, n_src, 0, P, *st, out,
                                     zb.ZERO_OUT_FULL, _hp(zb, t))
        torch.cuda.synchronize()
        out_ref, *ref = oracle.rs_adamw_reference(rows, n_src, *ref, HP_ORACLE, t)
        parity.assert_state(st, ref, what=f"t={t} ")
        assert np.array_equal(parity.bits(out), out_ref)
    too_many = [srcs[0]] * 65
    with pytest.raises(zb.ZeroError) as e:
        zb.zero_reduce_scatter_adamw(L, too_many, dt, 0, 65.0, 0, n_src, 0, P, *st, out,
                                     zb.ZERO_OUT_FULL, _hp(zb, 3))
    assert e.value.code == -3
