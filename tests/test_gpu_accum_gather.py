"""Parity of the accumulation kernels, the stage-3 gather and the ZeRO-3 per-unit
sequence against the oracle, through the C ABI."""
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


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("start", [0, 3])
def test_accumulate_local(zlib, cuda_device, dtype, start):
    zb = zlib
    N = 20_011
    L = zb.zero_layout([N], 1, align=1)
    rng = np.random.default_rng(11)
    acc = torch.zeros(N, device="cuda")
    ref = np.zeros(N, np.float32)
    for k in range(3):
        x = (rng.standard_normal(N) * 1e-3).astype(np.float32)
        if dtype == "bf16":
            xb = oracle.cast_bf16(x)
            src, code = inputs.from_bf16_bits(xb, "cuda"), zb.ZERO_BF16
            xr = oracle.bf16_to_f32(xb)
        else:
            src, code, xr = torch.from_numpy(x).cuda(), zb.ZERO_F32, x
        zb.zero_accumulate(L, zb.ZERO_ACC_LOCAL, [src], code, 0, acc, 0, start, N, k == 0)
        ref[start:] = xr[start:] if k == 0 else ref[start:] + xr[start:]
    torch.cuda.synchronize()
    parity.assert_bit_exact_f32(acc[start:], ref[start:])
    assert not parity.f32(acc)[:start].any()


@pytest.mark.parametrize("n_src", [1, 2, 3, 4, 8, 16, 64])
def test_accumulate_reduce(zlib, cuda_device, n_src):
    zb = zlib
    N = 8 * 2500 + 5
    L = zb.zero_layout([N], 1)
    g = inputs.grads_bf16(n_src, N, L.padded_n, seed=n_src, step=0)
    srcs = [g[r].cuda() for r in range(n_src)]
    A = torch.zeros(L.padded_n, device="cuda")
    ref = None
    for k in range(2):
        zb.zero_accumulate(L, zb.ZERO_ACC_REDUCE, srcs, zb.ZERO_BF16, 0, A, 0, 0, L.padded_n, k == 0)
        ref = oracle.accumulate_reduce(ref, parity.bits(g), first=(k == 0))
    torch.cuda.synchronize()
    parity.assert_bit_exact_f32(A, ref)


def test_accumulation_paths_small(zlib, cuda_device):
    """Gradient accumulation in small: n_dp = 4, K = 4 micro-batches; ZeRO-1
    (local fp32 accumulation, one reduce-scatter) and ZeRO-2 (reduce-scatter per
    micro-batch), each against its own oracle order, then against each other."""
    zb = zlib
    N, n_dp, K = 30_011, 4, 4
    L = zb.zero_layout([N], n_dp, bucket_elems=4096)
    P = L.padded_n
    w0 = inputs.master_weights(N, P, seed=4)
    s1 = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    s2 = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    o1 = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    o2 = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    acc = [torch.empty(P, device="cuda") for _ in range(n_dp)]
    A = torch.empty(P, device="cuda")
    micro = [inputs.grads_bf16(n_dp, N, P, seed=4, step=1, micro=k) for k in range(K)]
    for k, g in enumerate(micro):
        gd = [g[r].cuda() for r in range(n_dp)]
        zstep.zero1_accumulate_micro(L, gd, acc, first=(k == 0))
        zstep.zero2_accumulate_micro(L, gd, A, first=(k == 0))
    zstep.zero1_finish(L, acc, K, *s1, o1, _hp(zb, 1))
    zstep.zero2_finish(L, A, K, *s2, o2, _hp(zb, 1))
    torch.cuda.synchronize()
    # oracle, ZeRO-1 order
    acc_ref = [None] * n_dp
    for k, g in enumerate(micro):
        gb = parity.bits(g)
        for r in range(n_dp):
            acc_ref[r] = oracle.accumulate_local(acc_ref[r], gb[r], first=(k == 0))
    for r in range(n_dp):
        parity.assert_bit_exact_f32(acc[r], acc_ref[r])
    zero = np.zeros(P, np.float32)
    out1, *st1 = oracle.rs_adamw_reference(np.stack(acc_ref), n_dp * K, parity.f32(w0), zero, zero, HP, 1)
    parity.assert_state(s1, st1, what="zero1 ")
    assert np.array_equal(parity.bits(o1), out1)
    # oracle, ZeRO-2 order
    A_ref = None
    for k, g in enumerate(micro):
        A_ref = oracle.accumulate_reduce(A_ref, parity.bits(g), first=(k == 0))
    parity.assert_bit_exact_f32(A, A_ref)
    out2, *st2 = oracle.rs_adamw_reference(A_ref[None, :], n_dp * K, parity.f32(w0), zero, zero, HP, 1)
    parity.assert_state(s2, st2, what="zero2 ")
    assert np.array_equal(parity.bits(o2), out2)
    # the two orders: mean gradients agree within the fp32 summation bound
    x = np.stack([oracle.bf16_to_f32(parity.bits(g)).astype(np.float64) for g in micro])
    bound = (n_dp * K * 2.0 ** -24 / (1 - n_dp * K * 2.0 ** -24)) * np.abs(x).sum(axis=(0, 1))
    assert np.all(np.abs(np.stack(acc_ref).astype(np.float64).sum(0) - A_ref) <= 2 * bound + 1e-45)


@pytest.mark.parametrize("n_dp,S,align", [(1, 8, 8), (3, 5, 1), (8, 4096, 8), (7, 1001, 1), (65, 24, 8)])
def test_gather_is_concatenation(zlib, cuda_device, n_dp, S, align):
    zb = zlib
    L = zb.zero_layout([n_dp * S], n_dp, align=align)
    assert L.shard == S or align > 1
    rng = np.random.default_rng(n_dp)
    shards_np = rng.integers(0, 1 << 16, size=(n_dp, L.shard)).astype(np.uint16)
    shards = [inputs.from_bf16_bits(shards_np[o], "cuda") for o in range(n_dp)]
    full = torch.full((L.padded_n + 16,), 777, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    zb.zero_gather_layer(L, shards, full[: L.padded_n])
    torch.cuda.synchronize()
    fb = parity.bits(full)
    assert np.array_equal(fb[: L.padded_n], np.concatenate(list(shards_np)))
    assert np.all(fb[L.padded_n:] == 777)


def test_zero3_units(zlib, cuda_device):
    """The stage-3 sequence over ragged units (numel 1, 7, 4097, 33031 and a
    4-tensor block) at n_dp = 7: gather for forward, release, gather for
    backward, reduce-scatter the unit gradient, update the owned shards in bf16;
    at most two units resident; every gathered buffer is the concatenation of
    the shards; the reduce-scattered pieces equal the data-parallel gradient."""
    zb = zlib
    n_dp = 7
    units_numels = [[1], [7], [4097], [33_031], [1000, 24, 3, 5000]]
    units = []
    for i, numels in enumerate(units_numels):
        L = zb.zero_layout(numels, n_dp)
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=100 + i).cuda()
        shards = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
        shards.copy_(w)       # the initial bf16 weights: torch's cast (inputs only)
        units.append(zstep.Zero3Unit(L, shards.view(n_dp, L.shard), w,
                                     torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")))
    cap = max(u.layout.padded_n for u in units)
    ring = zstep.GatherRing(cap)
    ref_state = [[parity.f32(u.master), np.zeros(u.layout.padded_n, np.float32),
                  np.zeros(u.layout.padded_n, np.float32)] for u in units]
    ref_shards = [parity.bits(u.shards).copy() for u in units]
    # forward: gather each unit, "compute", release; the next unit's gather may overlap
    prev = None
    for i, u in enumerate(units):
        buf = zstep.zero3_gather(u, ring, ("fwd", i))
        torch.cuda.synchronize()
        assert np.array_equal(parity.bits(buf), ref_shards[i].reshape(-1))
        if prev is not None:
            ring.release(prev)
        prev = ("fwd", i)
        assert ring.resident <= 2
    ring.release(prev)
    # backward, in reverse: gather again, reduce-scatter the unit gradient, update
    for i in reversed(range(len(units))):
        u = units[i]
        L = u.layout
        buf = zstep.zero3_gather(u, ring, ("bwd", i))
        torch.cuda.synchronize()
        assert np.array_equal(parity.bits(buf), ref_shards[i].reshape(-1))
        g = inputs.grads_bf16(n_dp, L.n, L.padded_n, seed=200 + i, step=1)
        A = torch.empty(L.padded_n, device="cuda")
        zstep.zero3_layer_reduce_scatter(u, [g[r].cuda() for r in range(n_dp)], A)
        ring.release(("bwd", i))
        zstep.zero3_update(u, A, _hp(zb, 1))
        torch.cuda.synchronize()
        A_ref = oracle.accumulate_reduce(None, parity.bits(g), first=True)
        parity.assert_bit_exact_f32(A, A_ref)
        # each owner's piece of the mean is the data-parallel mean gradient's piece
        np.testing.assert_array_equal(A_ref / np.float32(n_dp), oracle.reduce_mean(parity.bits(g), n_dp))
        out_ref, *st = oracle.rs_adamw_reference(A_ref[None, :], n_dp, *ref_state[i], HP, 1)
        parity.assert_state([u.master, u.m, u.v], st, what=f"unit {i} ")
        assert np.array_equal(parity.bits(u.shards).reshape(-1), out_ref)
    assert ring.peak <= 2 and ring.resident == 0


@pytest.mark.parametrize("mode,n_src,dtype", [("local", 1, "bf16"), ("local", 1, "f32"),
                                              ("reduce", 1, "bf16"), ("reduce", 2, "bf16"),
                                              ("reduce", 4, "bf16"), ("reduce", 8, "bf16"),
                                              ("reduce", 2, "f32"), ("reduce", 5, "bf16")])
def test_accumulate_several_waves(zlib, cuda_device, mode, n_src, dtype):
    """5,000,011 elements: several passes of the multi-vector loops, a partial
    last group, a ragged tail; first and accumulating calls."""
    zb = zlib
    N = 5_000_011
    L = zb.zero_layout([N], 1, align=1)
    rng = np.random.default_rng(7 + n_src)
    dst = torch.zeros(N, device="cuda")
    ref = None
    for k in range(2):
        xf = (rng.standard_normal((n_src, N)) * 1e-3).astype(np.float32)
        if dtype == "bf16":
            xs = oracle.cast_bf16(xf)
            srcs = [inputs.from_bf16_bits(xs[r], "cuda") for r in range(n_src)]
            code = zb.ZERO_BF16
            xr = oracle.bf16_to_f32(xs)
        else:
            srcs = [torch.from_numpy(xf[r].copy()).cuda() for r in range(n_src)]
            code = zb.ZERO_F32
            xr = xf
        m = zb.ZERO_ACC_LOCAL if mode == "local" else zb.ZERO_ACC_REDUCE
        zb.zero_accumulate(L, m, srcs, code, 0, dst, 0, 0, N, k == 0)
        if mode == "local":
            ref = xr[0].copy() if k == 0 else ref + xr[0]
        elif dtype == "bf16":
            ref = oracle.accumulate_reduce(ref, xs, first=(k == 0))
        else:
            s = oracle.reduce_mean(xr, 1.0)        # the fp32 sum over sources (division by 1 is exact)
            ref = s if k == 0 else ref + s
    torch.cuda.synchronize()
    parity.assert_bit_exact_f32(dst, ref)


def test_gather_several_waves(zlib, cuda_device):
    zb = zlib
    n_dp, S = 3, 4_000_000
    L = zb.zero_layout([n_dp * S], n_dp)
    rng = np.random.default_rng(3)
    sh = rng.integers(0, 1 << 16, size=(n_dp, S)).astype(np.uint16)
    full = torch.empty(L.padded_n, dtype=torch.bfloat16, device="cuda")
    zb.zero_gather_layer(L, [inputs.from_bf16_bits(sh[o], "cuda") for o in range(n_dp)], full)
    torch.cuda.synchronize()
    assert np.array_equal(parity.bits(full), sh.reshape(-1))


def test_zero3_fused_reduce_scatter_update_equals_the_pair(zlib, cuda_device):
    """One micro-batch, no clipping: the fused per-unit reduce-scatter + update
    equals the layer reduce-scatter into fp32 followed by the update, bit for
    bit, on ragged units at n_dp = 7, over two steps."""
    zb = zlib
    n_dp = 7
    for i, numels in enumerate([[1], [4097], [33_031], [1000, 24, 3, 5000]]):
        L = zb.zero_layout(numels, n_dp)
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=500 + i).cuda()
        units = []
        for _ in range(2):
            shards = w.to(torch.bfloat16)
            units.append(zstep.Zero3Unit(L, shards.view(n_dp, L.shard), w.clone(),
                                         torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")))
        A = torch.empty(P, device="cuda")
        for t in (1, 2):
            g = inputs.grads_bf16(n_dp, L.n, P, seed=600 + i, step=t)
            gd = [g[r].cuda() for r in range(n_dp)]
            zstep.zero3_layer_reduce_scatter(units[0], gd, A)
            zstep.zero3_update(units[0], A, _hp(zb, t))
            zstep.zero3_reduce_scatter_update(units[1], gd, _hp(zb, t))
            torch.cuda.synchronize()
            for a, b in ((units[0].master, units[1].master), (units[0].m, units[1].m),
                         (units[0].v, units[1].v)):
                parity.assert_bit_exact_f32(a, parity.f32(b))
            assert torch.equal(units[0].shards.view(torch.int16), units[1].shards.view(torch.int16))


@pytest.mark.parametrize("int8", [False, True], ids=["bf16-gradients", "8-bit-gradients"])
def test_zero3_units_with_gradient_accumulation(zlib, cuda_device, int8):
    """Stage 3 with K = 3 micro-batches: each unit's layer reduce-scatter adds
    into its fp32 buffer (the first overwrites), and the update divides by
    n_dp * K -- bf16 gradients, or 8-bit gradients through the dequantizing
    reduce-scatter -- against the oracle on ragged units at n_dp = 5."""
    zb = zlib
    n_dp, K, block = 5, 3, 256
    for i, numels in enumerate([[7], [4097], [1000, 24, 3, 5000]]):
        L = zb.zero_layout(numels, n_dp)
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=1100 + i).cuda()
        unit = zstep.Zero3Unit(L, w.to(torch.bfloat16).view(n_dp, L.shard), w,
                               torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda"))
        w0 = parity.f32(w)
        A = torch.empty(P, device="cuda")
        A_ref = None
        for k in range(K):
            g = inputs.grads_bf16(n_dp, L.n, P, seed=1200 + i, step=1, micro=k)
            if int8:
                qg = zstep.Int8Grads(L, n_dp, block)
                qg.quantize([g[r].cuda() for r in range(n_dp)])
                zstep.zero3_layer_reduce_scatter_int8(unit, qg, A, first=(k == 0))
                q_ref, s_ref = oracle.quantize_grad_int8(parity.bits(g), n_dp, block)
                A_ref = oracle.accumulate_reduce_int8(A_ref, q_ref, s_ref, n_dp, block, k == 0)
            else:
                zstep.zero3_layer_reduce_scatter(unit, [g[r].cuda() for r in range(n_dp)], A, first=(k == 0))
                A_ref = oracle.accumulate_reduce(A_ref, parity.bits(g), first=(k == 0))
        zstep.zero3_update(unit, A, _hp(zb, 1), n_micro=K)
        torch.cuda.synchronize()
        parity.assert_bit_exact_f32(A, A_ref)
        z = np.zeros(P, np.float32)
        out_ref, *st = oracle.rs_adamw_reference(A_ref[None, :], n_dp * K, w0, z, z, HP, 1)
        parity.assert_state([unit.master, unit.m, unit.v], st, what=f"unit {i} ")
        assert np.array_equal(parity.bits(unit.shards).reshape(-1), out_ref)
