"""The fused update with an 8-bit output (zero_reduce_scatter_adamw_q8): the
owners' update writes their shards straight in the 8-bit block format.  It
must equal, bit for bit, the update into bf16 shards followed by
zero_quantize_int8 (block 256) -- and the oracle: its update, its bf16 cast and
its quantizer per shard."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

HP = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
BLOCK = 256


def _hp(zb, t):
    return zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, t)


def _unit(zb, numels, n_dp, seed):
    L = zb.zero_layout(numels, n_dp, align=BLOCK)
    P = L.padded_n
    w = inputs.master_weights(L.n, P, seed=seed).cuda()
    return zstep.Zero3Unit(L, w.to(torch.bfloat16).view(n_dp, L.shard), w,
                           torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda"))


def _clone(u):
    return zstep.Zero3Unit(u.layout, u.shards.clone(), u.master.clone(), u.m.clone(), u.v.clone())


def _oracle_codes(out_bits, n_dp, S):
    qs, ss = [], []
    for o in range(n_dp):
        q, s = oracle.quantize_int8(out_bits[o * S:(o + 1) * S], BLOCK)
        qs.append(q)
        ss.append(s)
    return np.concatenate(qs), np.concatenate(ss)


@pytest.mark.parametrize("numels,n_dp", [([1], 3), ([4097], 7), ([33_031], 8), ([1000, 24, 3, 5000], 8),
                                         ([300_000], 5)])
@pytest.mark.parametrize("fused_rs", [False, True], ids=["from-fp32-buffer", "from-bf16-gradients"])
def test_q8_update_matches_update_then_quantize_and_oracle(zlib, cuda_device, numels, n_dp, fused_rs):
    zb = zlib
    a = _unit(zb, numels, n_dp, seed=len(numels) + n_dp)
    b = _clone(a)
    L = a.layout
    P, S = L.padded_n, L.shard
    assert S % BLOCK == 0
    qa, qb = zstep.Int8Shards(L, BLOCK), zstep.Int8Shards(L, BLOCK)
    A = torch.empty(P, device="cuda")
    ref = [parity.f32(a.master), np.zeros(P, np.float32), np.zeros(P, np.float32)]
    for t in (1, 2):
        g = inputs.grads_bf16(n_dp, L.n, P, seed=50 + t, step=t, outlier_p=0.01)
        gd = [g[r].cuda() for r in range(n_dp)]
        # the pair: update into bf16 shards, then the quantizer
        zstep.zero3_layer_reduce_scatter(a, gd, A)
        zstep.zero3_update(a, A, _hp(zb, t))
        zstep.zero3_quantize(a, qa)
        # the fused path
        if fused_rs:
            zstep.zero3_reduce_scatter_update_q8(b, gd, qb, _hp(zb, t))
        else:
            A2 = torch.empty(P, device="cuda")
            zstep.zero3_layer_reduce_scatter(b, gd, A2)
            zstep.zero3_update_q8(b, A2, qb, _hp(zb, t))
        torch.cuda.synchronize()
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            parity.assert_bit_exact_f32(y, parity.f32(x))
        assert torch.equal(qa.q, qb.q) and torch.equal(qa.scales, qb.scales)
        # and the oracle
        out_ref, *ref = oracle.rs_adamw_reference(parity.bits(g), n_dp, *ref, HP, t)
        parity.assert_state([b.master, b.m, b.v], ref, what=f"t={t} ")
        q_ref, s_ref = _oracle_codes(out_ref, n_dp, S)
        np.testing.assert_array_equal(qb.q.cpu().numpy().reshape(-1), q_ref)
        np.testing.assert_array_equal(qb.scales[:, :qb.nb].cpu().numpy().reshape(-1), s_ref)


def test_q8_update_partial_owner_range(zlib, cuda_device):
    """Owners 2..4 of 6 and a range that starts and ends inside them on block
    boundaries: only that range's state, codes and scales change."""
    zb = zlib
    n_dp = 6
    u = _unit(zb, [50_000], n_dp, seed=9)
    L = u.layout
    P, S = L.padded_n, L.shard
    rb, re = 2, 5
    lo, hi = rb * S + 3 * BLOCK, re * S - 2 * BLOCK
    g = inputs.grads_bf16(n_dp, L.n, P, seed=3, step=1)
    gd = [g[r].cuda() for r in range(n_dp)]
    w = u.master[rb * S:re * S].clone()
    m = torch.zeros_like(w)
    v = torch.zeros_like(w)
    q = torch.full(((re - rb) * S,), 77, dtype=torch.int8, device="cuda")
    sc = torch.full(((re - rb) * S // BLOCK,), 5.0, device="cuda")
    zb.zero_reduce_scatter_adamw_q8(L, gd, zb.ZERO_BF16, 0, float(n_dp), rb, re, lo, hi, w, m, v, q, sc,
                                    BLOCK, _hp(zb, 1))
    torch.cuda.synchronize()
    z = np.zeros(P, np.float32)
    out_ref, w_ref, m_ref, v_ref = oracle.rs_adamw_reference(parity.bits(g), n_dp, parity.f32(u.master),
                                                             z, z, HP, 1)
    a, b = lo - rb * S, hi - rb * S
    parity.assert_bit_exact_f32(w[a:b], w_ref[lo:hi])
    parity.assert_bit_exact_f32(m[a:b], m_ref[lo:hi])
    qn, sn = q.cpu().numpy(), sc.cpu().numpy()
    for k in range(a // BLOCK, b // BLOCK):
        qk, sk = oracle.quantize_int8(out_ref[rb * S + k * BLOCK: rb * S + (k + 1) * BLOCK], BLOCK)
        assert np.array_equal(qn[k * BLOCK:(k + 1) * BLOCK], qk) and sn[k] == sk[0]
    assert np.all(qn[:a] == 77) and np.all(qn[b:] == 77)
    assert np.all(sn[:a // BLOCK] == 5.0) and np.all(sn[b // BLOCK:] == 5.0)
    assert torch.equal(w[:a], u.master[rb * S:rb * S + a]) and torch.equal(w[b:], u.master[rb * S + b:re * S])


@pytest.mark.parametrize("numels,n_dp", [([4097], 7), ([33_031], 8), ([1000, 24, 3, 5000], 3)])
def test_int8_gradient_update_with_8bit_output(zlib, cuda_device, numels, n_dp):
    """Both ZeRO++ 8-bit paths in one pass: from the ranks' 8-bit gradients
    straight to 8-bit shards.  Equal to the 8-bit accumulation into fp32, the
    update into bf16 and the quantizer, bit for bit, and to the oracle."""
    zb = zlib
    a = _unit(zb, numels, n_dp, seed=20 + n_dp)
    b = _clone(a)
    L = a.layout
    P, S = L.padded_n, L.shard
    qa, qb = zstep.Int8Shards(L, BLOCK), zstep.Int8Shards(L, BLOCK)
    A = torch.empty(P, device="cuda")
    ref = [parity.f32(a.master), np.zeros(P, np.float32), np.zeros(P, np.float32)]
    for t in (1, 2):
        g = inputs.grads_bf16(n_dp, L.n, P, seed=70 + t, step=t, outlier_p=0.01)
        qg = zstep.Int8Grads(L, n_dp, BLOCK)
        qg.quantize([g[r].cuda() for r in range(n_dp)])
        zstep.zero3_layer_reduce_scatter_int8(a, qg, A)
        zstep.zero3_update(a, A, _hp(zb, t))
        zstep.zero3_quantize(a, qa)
        zstep.zero3_reduce_scatter_update_int8_q8(b, qg, qb, _hp(zb, t))
        torch.cuda.synchronize()
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            parity.assert_bit_exact_f32(y, parity.f32(x))
        assert torch.equal(qa.q, qb.q) and torch.equal(qa.scales, qb.scales)
        q_ref, s_ref = oracle.quantize_grad_int8(parity.bits(g), n_dp, BLOCK)
        out_ref, *ref = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_dp, BLOCK, n_dp, *ref, HP, t)
        parity.assert_state([b.master, b.m, b.v], ref, what=f"t={t} ")
        cq, cs = _oracle_codes(out_ref, n_dp, S)
        np.testing.assert_array_equal(qb.q.cpu().numpy().reshape(-1), cq)
        np.testing.assert_array_equal(qb.scales[:, :qb.nb].cpu().numpy().reshape(-1), cs)


@pytest.mark.parametrize("n_dp", [1, 8])
def test_int8_gradient_update_with_8bit_output_state_off_the_32_byte_grid(zlib, cuda_device, n_dp):
    """The update from 8-bit gradients to 8-bit shards moves its fp32 state with
    256-bit accesses where every slice's state starts on a 32-byte boundary,
    and with 128-bit ones otherwise: state 32-byte aligned and state 16 bytes
    off that grid give the same bits, and both equal the oracle."""
    zb = zlib
    L = zb.zero_layout([33_031], n_dp, align=BLOCK)
    P, S = L.padded_n, L.shard
    w0 = inputs.master_weights(L.n, P, seed=91)
    g = inputs.grads_bf16(n_dp, L.n, P, seed=92, step=1, outlier_p=0.01)
    qg = zstep.Int8Grads(L, n_dp, BLOCK)
    qg.quantize([g[r].cuda() for r in range(n_dp)])
    qs, ss = qg.sources()
    q_ref, s_ref = oracle.quantize_grad_int8(parity.bits(g), n_dp, BLOCK)
    out_ref, *ref = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_dp, BLOCK, n_dp, parity.f32(w0),
                                                    np.zeros(P, np.float32), np.zeros(P, np.float32), HP, 1)
    cq, cs = _oracle_codes(out_ref, n_dp, S)
    results = []
    for off in (0, 4):                       # floats: 0 keeps the 32-byte grid, 4 is 16 bytes off it
        bufs = [torch.zeros(P + 8, device="cuda") for _ in range(3)]
        st = [b[off:off + P] for b in bufs]
        st[0].copy_(w0.cuda())
        assert st[0].data_ptr() % 32 == (0 if off == 0 else 16)
        q_out = torch.zeros(P, dtype=torch.int8, device="cuda")
        s_out = torch.zeros(P // BLOCK, device="cuda")
        zb.zero_reduce_scatter_adamw_int8_q8(L, qs, ss, BLOCK, float(n_dp), 0, n_dp, 0, P, *st, q_out, s_out,
                                             BLOCK, _hp(zb, 1))
        torch.cuda.synchronize()
        parity.assert_state(st, ref, what=f"offset {off} floats ")
        np.testing.assert_array_equal(q_out.cpu().numpy(), cq)
        np.testing.assert_array_equal(s_out.cpu().numpy(), cs)
        for b in bufs:                           # nothing written outside the state
            assert torch.count_nonzero(b[:off]) == 0 and torch.count_nonzero(b[off + P:]) == 0
        results.append([x.clone() for x in st] + [q_out, s_out])
    for x, y in zip(*results):
        assert torch.equal(x, y)
