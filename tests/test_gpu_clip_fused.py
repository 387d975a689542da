"""Parity of the fused accumulation finish (zero_accumulate_adamw), the global
gradient norm (zero_grad_norm_sq) and the clipped update
(zero_reduce_scatter_adamw_clip) against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

HP = oracle.AdamW()


def _hp(zb, t):
    return zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, t)


def _state(N, P, seed):
    w0 = inputs.master_weights(N, P, seed=seed)
    return w0, [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]


@pytest.mark.parametrize("n_dp,K,N", [(4, 4, 30_011), (2, 2, 9_999), (8, 3, 50_000), (3, 2, 12_345),
                                      (4, 2, 2_000_003)])
def test_fused_finish_equals_unfused_and_oracle(zlib, cuda_device, n_dp, K, N):
    zb = zlib
    L = zb.zero_layout([N], n_dp, bucket_elems=1 << 20)
    P = L.padded_n
    micro = [inputs.grads_bf16(n_dp, N, P, seed=n_dp, step=1, micro=k) for k in range(K)]
    mdev = [[g[r].cuda() for r in range(n_dp)] for g in micro]
    w0, s_u1 = _state(N, P, 1)
    _, s_f1 = _state(N, P, 1)
    _, s_u2 = _state(N, P, 1)
    _, s_f2 = _state(N, P, 1)
    outs = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    acc = [torch.empty(P, device="cuda") for _ in range(n_dp)]
    A = torch.empty(P, device="cuda")
    # stage 1: K-1 micro-batches accumulated, the last one fused
    for k in range(K - 1):
        zstep.zero1_accumulate_micro(L, mdev[k], acc, first=(k == 0))
    acc_before = [a.clone() for a in acc]
    zstep.zero1_finish_fused(L, acc, mdev[-1], K, *s_f1, outs[0], _hp(zb, 1))
    for r in range(n_dp):      # the fused finish reads the accumulators only
        assert torch.equal(acc[r], acc_before[r])
    zstep.zero1_accumulate_micro(L, mdev[-1], acc, first=False)
    zstep.zero1_finish(L, acc, K, *s_u1, outs[1], _hp(zb, 1))
    # stage 2
    for k in range(K - 1):
        zstep.zero2_accumulate_micro(L, mdev[k], A, first=(k == 0))
    zstep.zero2_finish_fused(L, A, mdev[-1], K, *s_f2, outs[2], _hp(zb, 1))
    zstep.zero2_accumulate_micro(L, mdev[-1], A, first=False)
    zstep.zero2_finish(L, A, K, *s_u2, outs[3], _hp(zb, 1))
    torch.cuda.synchronize()
    for fused, unfused in ((s_f1, s_u1), (s_f2, s_u2)):
        for a, b in zip(fused, unfused):
            parity.assert_bit_exact_f32(a, b)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[2].view(torch.int16), outs[3].view(torch.int16))
    # against the oracle's two orders
    acc_ref = [None] * n_dp
    A_ref = None
    for k, g in enumerate(micro):
        gb = parity.bits(g)
        for r in range(n_dp):
            acc_ref[r] = oracle.accumulate_local(acc_ref[r], gb[r], first=(k == 0))
        A_ref = oracle.accumulate_reduce(A_ref, gb, first=(k == 0))
    z = np.zeros(P, np.float32)
    o1, *st1 = oracle.rs_adamw_reference(np.stack(acc_ref), n_dp * K, parity.f32(w0), z, z, HP, 1)
    o2, *st2 = oracle.rs_adamw_reference(A_ref[None, :], n_dp * K, parity.f32(w0), z, z, HP, 1)
    parity.assert_state(s_f1, st1, what="zero1 fused ")
    parity.assert_state(s_f2, st2, what="zero2 fused ")
    assert np.array_equal(parity.bits(outs[0]), o1) and np.array_equal(parity.bits(outs[2]), o2)


def test_fused_finish_misaligned_range(zlib, cuda_device):
    zb = zlib
    N, n_dp = 5_003, 4
    L = zb.zero_layout([N], 1, align=1)
    g = inputs.grads_bf16(n_dp, N, N, seed=3, step=1)
    gd = [g[r].cuda() for r in range(n_dp)]
    rng = np.random.default_rng(0)
    accs = (rng.standard_normal((n_dp, N)) * 1e-3).astype(np.float32)
    acc = [torch.from_numpy(accs[r].copy()).cuda() for r in range(n_dp)]
    w0, st = _state(N, N, 2)
    out = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    start = 3
    zb.zero_accumulate_adamw(L, zb.ZERO_ACC_LOCAL, acc, 0, gd, 0, float(n_dp * 2), 0, 1, start, N,
                             *st, out, zb.ZERO_OUT_FULL, _hp(zb, 5))
    torch.cuda.synchronize()
    fin = np.stack([oracle.accumulate_local(accs[r], parity.bits(g)[r], first=False)
                    for r in range(n_dp)])
    z = np.zeros(N - start, np.float32)
    ref_out, *ref = oracle.rs_adamw_reference(fin[:, start:], n_dp * 2, parity.f32(w0)[start:], z, z,
                                              HP, 5)
    parity.assert_state([x[start:] for x in st], ref)
    assert np.array_equal(parity.bits(out)[start:], ref_out)


@pytest.mark.parametrize("n_src,dtype,N", [(8, "bf16", 100_003), (4, "bf16", 77_777), (1, "f32", 64_000),
                                           (3, "bf16", 33_333), (2, "f32", 5_000_011), (8, "bf16", 7)])
def test_grad_norm_sq(zlib, cuda_device, n_src, dtype, N):
    zb = zlib
    L = zb.zero_layout([N], 1, align=1)
    rng = np.random.default_rng(n_src * 7 + N)
    xf = (rng.standard_normal((n_src, N)) * 1e-2).astype(np.float32)
    if dtype == "bf16":
        src_np = oracle.cast_bf16(xf)
        srcs = [inputs.from_bf16_bits(src_np[r], "cuda") for r in range(n_src)]
        code = zb.ZERO_BF16
    else:
        src_np = xf
        srcs = [torch.from_numpy(xf[r].copy()).cuda() for r in range(n_src)]
        code = zb.ZERO_F32
    bufs = zstep.NormBuffers("cuda")
    ref = oracle.grad_norm_sq(src_np, n_src)
    zb.zero_grad_norm_sq(L, srcs, code, 0, float(n_src), 0, N, bufs.workspace, bufs.norm_sq, False)
    got = float(bufs.norm_sq.item())
    assert got == pytest.approx(ref, rel=1e-12)
    # the same over three pieces, accumulated, and over a misaligned start
    cuts = [0, N // 3, (2 * N) // 3 + 1, N]
    for j in range(3):
        zb.zero_grad_norm_sq(L, srcs, code, 0, float(n_src), cuts[j], cuts[j + 1], bufs.workspace,
                             bufs.norm_sq, j > 0)
    assert float(bufs.norm_sq.item()) == pytest.approx(ref, rel=1e-12)
    # repeated calls give the same bits
    zb.zero_grad_norm_sq(L, srcs, code, 0, float(n_src), 0, N, bufs.workspace, bufs.norm_sq, False)
    assert float(bufs.norm_sq.item()) == got
    # an empty range writes 0
    zb.zero_grad_norm_sq(L, srcs, code, 0, float(n_src), 5, 5, bufs.workspace, bufs.norm_sq, False)
    assert float(bufs.norm_sq.item()) == 0.0


def test_grad_norm_workspace_too_small(zlib, cuda_device):
    zb = zlib
    L = zb.zero_layout([1024], 1)
    src = [torch.zeros(1024, dtype=torch.bfloat16, device="cuda")]
    small = torch.empty(4, dtype=torch.float64, device="cuda")
    nsq = torch.zeros(1, dtype=torch.float64, device="cuda")
    with pytest.raises(zb.ZeroError) as e:
        zb.zero_grad_norm_sq(L, src, zb.ZERO_BF16, 0, 1.0, 0, 1024, small, nsq, False)
    assert e.value.code == zb.ZERO_ERANGE


@pytest.mark.parametrize("std,max_norm", [(1.0, 1.0), (1e-3, 1.0), (3e-2, 0.5)])
def test_clipped_step(zlib, cuda_device, std, max_norm):
    """ZeRO-2 step with clipping, n_dp = 4, several buckets: active clipping
    (std 1), inactive (std 1e-3: coefficient exactly 1, the step equals the
    unclipped one bit for bit), and a threshold of 0.5."""
    zb = zlib
    N, n_dp = 100_003, 4
    L = zb.zero_layout([N], n_dp, bucket_elems=30_000)
    P = L.padded_n
    g = inputs.grads_bf16(n_dp, N, P, seed=11, step=1, std=std)
    gd = [g[r].cuda() for r in range(n_dp)]
    w0, st = _state(N, P, 4)
    _, st_u = _state(N, P, 4)
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    out_u = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    bufs = zstep.NormBuffers("cuda")
    zstep.zero12_step_clipped(L, gd, *st, out, _hp(zb, 1), max_norm, bufs)
    zstep.zero12_step(L, gd, *st_u, out_u, _hp(zb, 1))
    torch.cuda.synchronize()
    gb = parity.bits(g)
    ref_nsq = oracle.grad_norm_sq(gb, n_dp)
    gpu_nsq = float(bufs.norm_sq.item())
    assert gpu_nsq == pytest.approx(ref_nsq, rel=1e-12)
    coef = oracle.clip_coef(ref_nsq, max_norm)
    assert oracle.clip_coef(gpu_nsq, max_norm) == coef
    z = np.zeros(P, np.float32)
    ref_out, *ref = oracle.rs_adamw_reference(gb, n_dp, parity.f32(w0), z, z, HP, 1,
                                              clip=(ref_nsq, max_norm))
    parity.assert_state(st, ref)
    assert np.array_equal(parity.bits(out), ref_out)
    if coef == np.float32(1.0):
        for a, b in zip(st, st_u):
            parity.assert_bit_exact_f32(a, b)
    else:
        assert coef < 1.0


def test_grad_norm_extreme_values(zlib, cuda_device):
    """Squares outside the fp32 pair's exact range (|g| < 2^-50 or >= 2^60)
    take the fp64 path: tiny, huge, zero and ordinary values mixed."""
    zb = zlib
    N = 40_000
    L = zb.zero_layout([N], 1, align=1)
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((2, N)) * 1e-3).astype(np.float32)
    x[:, :1000] = 1e-20
    x[:, 1000:1010] = 3e25
    x[:, 1010:2000] = 0.0
    x[0, 2000:2100] = 2.0 ** -50
    x[1, 2000:2100] = 0.0
    srcs = [torch.from_numpy(x[r].copy()).cuda() for r in range(2)]
    bufs = zstep.NormBuffers("cuda")
    zb.zero_grad_norm_sq(L, srcs, zb.ZERO_F32, 0, 2.0, 0, N, bufs.workspace, bufs.norm_sq, False)
    assert float(bufs.norm_sq.item()) == pytest.approx(oracle.grad_norm_sq(x, 2.0), rel=1e-12)
    # only tiny values: the answer comes from the fp64 path alone
    t = np.full((1, 4096), 1e-25, np.float32)
    zb.zero_grad_norm_sq(L, [torch.from_numpy(t[0].copy()).cuda()], zb.ZERO_F32, 0, 1.0, 0, 4096,
                         bufs.workspace, bufs.norm_sq, False)
    assert float(bufs.norm_sq.item()) == pytest.approx(oracle.grad_norm_sq(t, 1.0), rel=1e-12)


@pytest.mark.parametrize("std,max_norm", [(1.0, 1.0), (1e-3, 1.0)])
def test_zero3_clipped_units(zlib, cuda_device, std, max_norm):
    """Stage 3 with clipping: every unit's gradient is reduce-scattered into
    fp32, the squared norm of the mean gradient accumulates over all units on
    the device, then every unit updates with the clipped gradient (ragged units,
    n_dp = 7; active clipping at std 1, coefficient 1 at std 1e-3)."""
    zb = zlib
    n_dp = 7
    units, As, gs, refs = [], [], [], []
    for i, numels in enumerate([[1], [4097], [33_031], [1000, 24, 3, 5000]]):
        L = zb.zero_layout(numels, n_dp)
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=800 + i).cuda()
        u = zstep.Zero3Unit(L, w.to(torch.bfloat16).view(n_dp, L.shard), w,
                            torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda"))
        g = inputs.grads_bf16(n_dp, L.n, P, seed=900 + i, step=1, std=std)
        A = torch.empty(P, device="cuda")
        zstep.zero3_layer_reduce_scatter(u, [g[r].cuda() for r in range(n_dp)], A)
        units.append(u)
        As.append(A)
        gs.append(g)
        refs.append(parity.f32(w))
    bufs = zstep.NormBuffers("cuda")
    zstep.zero3_clipped_updates(units, As, _hp(zb, 1), max_norm, bufs)
    torch.cuda.synchronize()
    A_refs = [oracle.accumulate_reduce(None, parity.bits(g), True) for g in gs]
    nsq_ref = sum(oracle.grad_norm_sq(A[None, :], n_dp) for A in A_refs)
    gpu_nsq = float(bufs.norm_sq.item())
    assert gpu_nsq == pytest.approx(nsq_ref, rel=1e-12)
    coef = oracle.clip_coef(nsq_ref, max_norm)
    assert oracle.clip_coef(gpu_nsq, max_norm) == coef
    assert (coef < 1.0) == (std == 1.0)
    for u, A_ref, w0 in zip(units, A_refs, refs):
        z = np.zeros(A_ref.size, np.float32)
        out_ref, *st = oracle.rs_adamw_reference(A_ref[None, :], n_dp, w0, z, z, HP, 1,
                                                 clip=(nsq_ref, max_norm))
        parity.assert_state([u.master, u.m, u.v], st)
        assert np.array_equal(parity.bits(u.shards).reshape(-1), out_ref)
