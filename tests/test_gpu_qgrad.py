"""Parity of the 8-bit gradient reduce-scatter (ZeRO++ quantized gradients:
zero_quantize_int8 over each rank's gradient, zero_reduce_scatter_adamw_int8,
zero_accumulate_int8) with the oracle, bit for bit, through the C ABI."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

HP = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


def _hp(zb, t):
    return zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, t)


def _quantized(zb, L, g_cpu, block):
    """Quantize every rank's gradient on the GPU; check codes and scales
    against the oracle; return (Int8Grads, oracle codes, oracle scales)."""
    qg = zstep.Int8Grads(L, g_cpu.shape[0], block)
    qg.quantize([g_cpu[r].cuda() for r in range(g_cpu.shape[0])])
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_grad_int8(parity.bits(g_cpu), L.n_dp, block)
    np.testing.assert_array_equal(qg.q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(qg.scales[:, :L.n_dp * qg.nb].cpu().numpy(), s_ref)
    return qg, q_ref, s_ref


@pytest.mark.parametrize("N,n_dp,align,bucket,block", [
    (1 << 20, 4, 8, 500_000_000, 256),      # the tiny configuration's sizes
    (100_003, 3, 8, 30_000, 256),           # buckets crossing owners, ragged
    (65_541, 8, 8, 20_000, 512),
    (300_007, 16, 8, 500_000_000, 2048),    # 16 sources, blocks longer than a slice's tail
    (4097, 5, 1, 1000, 256),                # S = 820: slices off the 8-element grid
    (7, 2, 1, 500_000_000, 256),            # fewer elements than one vector
    (50_000, 6, 8, 500_000_000, 1024),      # 6 sources: the runtime-count kernel
    (64_005, 64, 8, 500_000_000, 256),      # the most sources a call takes
])
def test_step_matches_oracle(zlib, cuda_device, N, n_dp, align, bucket, block):
    """Two steps of quantize + fused update against the oracle: codes, scales,
    fp32 state and the bf16 output all bit-exact."""
    zb = zlib
    L = zb.zero_layout([N], n_dp, align=align, bucket_elems=bucket)
    P = L.padded_n
    w0 = inputs.master_weights(N, P, seed=n_dp)
    st = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    ref = [parity.f32(w0), np.zeros(P, np.float32), np.zeros(P, np.float32)]
    for t in (1, 2):
        g = inputs.grads_bf16(n_dp, N, P, seed=n_dp, step=t, outlier_p=0.01)
        qg, q_ref, s_ref = _quantized(zb, L, g, block)
        zstep.zero12_step_int8(L, qg, *st, out, _hp(zb, t))
        torch.cuda.synchronize()
        out_ref, *ref = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_dp, block, n_dp, *ref, HP, t)
        parity.assert_state(st, ref, what=f"t={t} ")
        assert np.array_equal(parity.bits(out), out_ref)


def test_partial_range_shard_output(zlib, cuda_device):
    """Owners 1..2 of 4, a range from S + 5 to 3S - 3 (off the 8-element grid at
    both ends, crossing one owner boundary), bf16 into the owners' own shards:
    exactly the range changes, and it matches the oracle."""
    zb = zlib
    N, n_dp, block = 40_000, 4, 256
    L = zb.zero_layout([N], n_dp)
    S, P = L.shard, L.padded_n
    g = inputs.grads_bf16(n_dp, N, P, seed=5, step=1)
    qg, q_ref, s_ref = _quantized(zb, L, g, block)
    w0 = inputs.master_weights(N, P, seed=5)
    w = w0[S:3 * S].clone().cuda()
    m = torch.zeros(2 * S, device="cuda")
    v = torch.zeros(2 * S, device="cuda")
    out = torch.full((2 * S,), 3.0, dtype=torch.bfloat16, device="cuda")
    begin, end = S + 5, 3 * S - 3
    qs, ss = qg.sources()
    zb.zero_reduce_scatter_adamw_int8(L, qs, ss, block, float(n_dp), 1, 3, begin, end, w, m, v, out,
                                      zb.ZERO_OUT_SHARD, _hp(zb, 1))
    torch.cuda.synchronize()
    z = np.zeros(P, np.float32)
    out_ref, w_ref, m_ref, v_ref = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_dp, block, n_dp,
                                                                    parity.f32(w0), z, z, HP, 1)
    sel = slice(begin - S, end - S)
    for got, full, init in ((w, w_ref, parity.f32(w0)[S:3 * S]), (m, m_ref, np.zeros(2 * S, np.float32)),
                            (v, v_ref, np.zeros(2 * S, np.float32))):
        x = parity.f32(got)
        parity.assert_bit_exact_f32(x[sel], full[begin:end])
        assert np.array_equal(x[:5], init[:5]) and np.array_equal(x[-3:], init[-3:])
    ob = parity.bits(out)
    assert np.array_equal(ob[sel], out_ref[begin:end])
    three = oracle.cast_bf16(np.array([3.0], np.float32))[0]
    assert np.all(ob[:5] == three) and np.all(ob[-3:] == three)


@pytest.mark.parametrize("n_dp,block", [(8, 256), (4, 512), (3, 256), (1, 2048)])
def test_accumulate_overwrite_then_add(zlib, cuda_device, n_dp, block):
    """The owners' fp32 accumulation of two micro-batches of 8-bit gradients,
    over the whole vector (dst_base 0) and over one owner's slice alone
    (dst_base = o*S, a buffer of S elements)."""
    zb = zlib
    N = 123_457
    L = zb.zero_layout([N], n_dp)
    S, P = L.shard, L.padded_n
    A = torch.empty(P, device="cuda")
    o = n_dp // 2
    Ao = torch.empty(S, device="cuda")
    ref = None
    for k in range(2):
        g = inputs.grads_bf16(n_dp, N, P, seed=9, step=1, micro=k)
        qg, q_ref, s_ref = _quantized(zb, L, g, block)
        qs, ss = qg.sources()
        zb.zero_accumulate_int8(L, qs, ss, block, A, 0, 0, P, k == 0)
        zb.zero_accumulate_int8(L, qs, ss, block, Ao, o * S, o * S, (o + 1) * S, k == 0)
        torch.cuda.synchronize()
        ref = oracle.accumulate_reduce_int8(ref, q_ref, s_ref, n_dp, block, k == 0)
        parity.assert_bit_exact_f32(A, ref)
        parity.assert_bit_exact_f32(Ao, ref[o * S:(o + 1) * S])


def test_zero3_units_with_int8_gradients(zlib, cuda_device):
    """The stage-3 backward over ragged units with 8-bit gradients: quantize
    each rank's unit gradient, reduce-scatter into fp32, update the owned
    shards in bf16 -- bit-exact against the oracle."""
    zb = zlib
    n_dp, block = 7, 256
    for i, numels in enumerate([[1], [4097], [33_031], [1000, 24, 3, 5000]]):
        L = zb.zero_layout(numels, n_dp)
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=300 + i).cuda()
        shards = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
        unit = zstep.Zero3Unit(L, shards.view(n_dp, L.shard), w, torch.zeros(P, device="cuda"),
                               torch.zeros(P, device="cuda"))
        w_ref = parity.f32(w)
        g = inputs.grads_bf16(n_dp, L.n, P, seed=400 + i, step=1)
        qg, q_ref, s_ref = _quantized(zb, L, g, block)
        A = torch.empty(P, device="cuda")
        zstep.zero3_layer_reduce_scatter_int8(unit, qg, A)
        zstep.zero3_update(unit, A, _hp(zb, 1))
        torch.cuda.synchronize()
        A_ref = oracle.accumulate_reduce_int8(None, q_ref, s_ref, n_dp, block, True)
        parity.assert_bit_exact_f32(A, A_ref)
        z = np.zeros(P, np.float32)
        out_ref, *st = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_dp, block, n_dp, w_ref, z, z,
                                                       HP, 1)
        parity.assert_state([unit.master, unit.m, unit.v], st, what=f"unit {i} ")
        assert np.array_equal(parity.bits(unit.shards).reshape(-1), out_ref)


def test_argument_errors(zlib, cuda_device):
    zb = zlib
    L = zb.zero_layout([4096], 2)
    P = L.padded_n
    g = inputs.grads_bf16(2, 4096, P, seed=1, step=1)
    qg = zstep.Int8Grads(L, 2, 256)
    qg.quantize([g[r].cuda() for r in range(2)])
    qs, ss = qg.sources()
    st = [torch.zeros(P, device="cuda") for _ in range(3)]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    qa, sa = _raw_sources(qs, ss)
    rc = zb.load().zero_reduce_scatter_adamw_int8(                # block not in the format
        ctypes.byref(L), qa, sa, 2, 128, 2.0, 0, 2, 0, P, *[x.data_ptr() for x in st],
        out.data_ptr(), zb.ZERO_OUT_FULL, ctypes.byref(_hp(zb, 1)), None)
    assert rc == -1
    with pytest.raises(zb.ZeroError) as e:                      # range outside the owners
        zb.zero_reduce_scatter_adamw_int8(L, qs, ss, 256, 2.0, 1, 2, 0, P, *st, out,
                                          zb.ZERO_OUT_FULL, _hp(zb, 1))
    assert e.value.code == -1
    # dst off the 16-byte grid runs the element kernel, with the same result
    A = torch.empty(P, device="cuda")
    A_off = torch.empty(P + 1, device="cuda")[1:]
    zb.zero_accumulate_int8(L, qs, ss, 256, A, 0, 0, P, True)
    zb.zero_accumulate_int8(L, qs, ss, 256, A_off, 0, 0, P, True)
    torch.cuda.synchronize()
    parity.assert_bit_exact_f32(A_off, parity.f32(A))
    # dst not 4-byte aligned is refused before any launch
    raw = torch.zeros(4 * P + 8, dtype=torch.uint8, device="cuda")
    rc = zb.load().zero_accumulate_int8(ctypes.byref(L), qa, sa, 2, 256, raw.data_ptr() + 2, 0, 0,
                                        P, 1, None)
    assert rc == -2
    zb.zero_status_check()


def _raw_sources(qs, ss):
    n = len(qs)
    return ((ctypes.c_void_p * n)(*[x.data_ptr() for x in qs]),
            (ctypes.c_void_p * n)(*[x.data_ptr() for x in ss]))


def test_whole_shards_of_later_owners(zlib, cuda_device):
    """Owners 1 and 2 of 4 over exactly their shards [S, 3S) -- one launch over
    both slices starting at owner 1: the update into the owners' own shards,
    the update with 8-bit output, and the accumulation into a buffer based at S,
    each bit-exact against the oracle and writing nothing outside its range."""
    zb = zlib
    N, n_dp, block = 60_000, 4, 256
    L = zb.zero_layout([N], n_dp, align=256)
    S, P = L.shard, L.padded_n
    g = inputs.grads_bf16(n_dp, N, P, seed=13, step=1)
    qg, q_ref, s_ref = _quantized(zb, L, g, block)
    qs, ss = qg.sources()
    w0 = inputs.master_weights(N, P, seed=13)
    z = np.zeros(P, np.float32)
    out_ref, w_ref, m_ref, v_ref = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_dp, block, n_dp,
                                                                    parity.f32(w0), z, z, HP, 1)
    sel = slice(S, 3 * S)
    # bf16 into the owners' shards; 16-byte guard bands keep every buffer aligned
    # for the vector kernel, so the call takes the one-launch path
    bufs = [torch.full((2 * S + 8,), 7.0, device="cuda") for _ in range(3)]
    bufs[0][4:-4] = w0[sel].cuda()
    bufs[1][4:-4] = 0.0
    bufs[2][4:-4] = 0.0
    out = torch.full((2 * S + 16,), 5.0, dtype=torch.bfloat16, device="cuda")
    zb.zero_reduce_scatter_adamw_int8(L, qs, ss, block, float(n_dp), 1, 3, S, 3 * S, bufs[0][4:-4],
                                      bufs[1][4:-4], bufs[2][4:-4], out[8:-8], zb.ZERO_OUT_SHARD, _hp(zb, 1))
    # the 8-bit output
    w8 = w0[sel].clone().cuda()
    m8, v8 = torch.zeros(2 * S, device="cuda"), torch.zeros(2 * S, device="cuda")
    q8 = torch.zeros(2 * S + 32, dtype=torch.int8, device="cuda")
    s8 = torch.full((2 * S // 256 + 2,), 9.0, device="cuda")
    zb.zero_reduce_scatter_adamw_int8_q8(L, qs, ss, block, float(n_dp), 1, 3, S, 3 * S, w8, m8, v8,
                                         q8[16:-16], s8[1:-1], 256, _hp(zb, 1))
    # the accumulation into a buffer of 2S elements based at flat S
    A = torch.full((2 * S + 8,), 11.0, device="cuda")
    zb.zero_accumulate_int8(L, qs, ss, block, A[4:-4], S, S, 3 * S, True)
    torch.cuda.synchronize()
    for got, ref in zip(bufs, (w_ref, m_ref, v_ref)):
        x = parity.f32(got)
        parity.assert_bit_exact_f32(x[4:-4], ref[sel])
        assert (x[:4] == 7.0).all() and (x[-4:] == 7.0).all()
    ob = parity.bits(out)
    assert np.array_equal(ob[8:-8], out_ref[sel])
    five = oracle.cast_bf16(np.array([5.0], np.float32))[0]
    assert (ob[:8] == five).all() and (ob[-8:] == five).all()
    parity.assert_bit_exact_f32(w8, w_ref[sel])
    for o in range(2):
        qo, so = oracle.quantize_int8(out_ref[(1 + o) * S:(2 + o) * S], 256)
        assert np.array_equal(q8[16 + o * S:16 + (o + 1) * S].cpu().numpy(), qo)
        assert np.array_equal(s8[1 + o * (S // 256):1 + (o + 1) * (S // 256)].cpu().numpy(), so)
    assert (q8[:16] == 0).all() and (q8[-16:] == 0).all() and s8[0] == 9.0 and s8[-1] == 9.0
    A_ref = oracle.accumulate_reduce_int8(None, q_ref, s_ref, n_dp, block, True)
    a = parity.f32(A)
    parity.assert_bit_exact_f32(a[4:-4], A_ref[sel])
    assert (a[:4] == 11.0).all() and (a[-4:] == 11.0).all()
