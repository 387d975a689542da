"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times.  Every element's update depends only on that element's own
inputs, so the oracle is run on sampled elements (random positions plus every
bucket and shard boundary, the first and last elements and the padding) and
compared one by one; properties that hold at any size are checked on every
element on the device (the bf16 buffer is the cast of the master weights, the
padding stays zero, nothing became non-finite)."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HP = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
SEED = 0


def _hp(zb, t):
    return zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, t)


def _sample_indices(lo, hi, boundaries, n_random=1 << 18, seed=0):
    rng = np.random.default_rng(seed)
    idx = [rng.integers(lo, hi, size=n_random)]
    for b in boundaries:
        idx.append(np.arange(b - 8, b + 8))
    idx.append(np.arange(lo, lo + 64))
    idx.append(np.arange(hi - 64, hi))
    idx = np.unique(np.concatenate(idx))
    return idx[(idx >= lo) & (idx < hi)]


def _take(t, idx_dev):
    return t.index_select(0, idx_dev)


def _bits_at(t, idx_dev):
    return parity.bits(_take(t, idx_dev))


def _full_properties(master, out_slice, n_real_in_slice):
    """On the device, over every element: out is the RNE cast of master, the
    padding is zero and nothing is non-finite."""
    assert torch.isfinite(master).all()
    cast = master.to(torch.bfloat16)   # torch's own round-to-nearest-even cast
    assert torch.equal(out_slice.view(torch.int16), cast.view(torch.int16))
    if n_real_in_slice < master.numel():
        assert not master[n_real_in_slice:].any()
        assert not out_slice[n_real_in_slice:].view(torch.int16).any()


def test_gpt2xl_zero2_all_shards(zlib, cuda_device):
    """GPT-2-XL shapes (N = 1,557,611,200), n_dp = 8, 5e8-element buckets,
    all eight owned shards updated per step, 5 steps (the later ones with
    non-zero moments)."""
    zb = zlib
    dev = cuda_device
    L = zb.zero_layout(inputs.gpt2xl_numels(), 8, 8, 500_000_000)
    P, S = L.padded_n, L.shard
    assert (L.n, P, L.n_buckets) == (1_557_611_200, 1_557_611_200, 4)
    g = torch.empty((8, P), dtype=torch.bfloat16, device=dev)
    master = inputs.master_weights(L.n, P, seed=SEED, device=dev)
    m = torch.zeros(P, device=dev)
    v = torch.zeros(P, device=dev)
    out = torch.zeros(P, dtype=torch.bfloat16, device=dev)
    bounds = [b * L.bucket for b in range(1, L.n_buckets)] + [o * S for o in range(1, 8)]
    idx = _sample_indices(0, P, bounds)
    idx_dev = torch.from_numpy(idx).to(dev)
    ref = [parity.f32(_take(x, idx_dev)) for x in (master, m, v)]
    for t in range(1, 6):
        for r in range(8):
            inputs.grad_bf16_into(g[r], L.n, SEED, step=t, rank=r)
        gs = np.stack([_bits_at(g[r], idx_dev) for r in range(8)])
        zstep.zero12_step(L, [g[r] for r in range(8)], master, m, v, out, _hp(zb, t))
        zb.zero_status_check()
        ref_out, *ref = oracle.rs_adamw_reference(gs, 8, *ref, HP, t)
        parity.assert_state([_take(x, idx_dev) for x in (master, m, v)], ref, what=f"t={t} ")
        assert np.array_equal(_bits_at(out, idx_dev), ref_out)
    _full_properties(master, out, L.n)


def test_llama7b_one_shard(zlib, cuda_device):
    """Llama-7B shapes (N = 6,738,415,616) at n_dp = 8: one owned shard of
    842,301,952 elements, 8 bf16 gradient slices with 1 % outliers x100, the
    fused update writing into the full bf16 buffer, 5 steps."""
    zb = zlib
    dev = cuda_device
    L = zb.zero_layout(inputs.llama7b_numels(), 8, 8, 500_000_000)
    S = L.shard
    assert S == 842_301_952
    o = 3
    lo, hi = o * S, (o + 1) * S
    g = torch.empty((8, S), dtype=torch.bfloat16, device=dev)
    master = inputs.master_weights(S, S, seed=SEED, device=dev)
    m = torch.zeros(S, device=dev)
    v = torch.zeros(S, device=dev)
    out = torch.full((L.padded_n,), 0x1234, dtype=torch.int16, device=dev).view(torch.bfloat16)
    bounds = [b * L.bucket - lo for b in range(1, L.n_buckets) if lo < b * L.bucket < hi]
    idx = _sample_indices(0, S, bounds, seed=1)
    idx_dev = torch.from_numpy(idx).to(dev)
    ref = [parity.f32(_take(x, idx_dev)) for x in (master, m, v)]
    for t in range(1, 6):
        for r in range(8):
            inputs.grad_bf16_into(g[r], S, SEED, step=t, rank=r, outlier_p=0.01)
        gs = np.stack([_bits_at(g[r], idx_dev) for r in range(8)])
        zstep.zero12_step(L, [g[r] for r in range(8)], master, m, v, out, _hp(zb, t),
                          rank_begin=o, rank_end=o + 1, grad_base=lo)
        zb.zero_status_check()
        ref_out, *ref = oracle.rs_adamw_reference(gs, 8, *ref, HP, t)
        parity.assert_state([_take(x, idx_dev) for x in (master, m, v)], ref, what=f"t={t} ")
        assert np.array_equal(_bits_at(out[lo:hi], idx_dev), ref_out)
    _full_properties(master, out[lo:hi], S)
    # nothing outside the owner's part of the full buffer was written
    iv = out.view(torch.int16)
    assert bool((iv[:lo] == 0x1234).all()) and bool((iv[hi:] == 0x1234).all())


def test_gpt2xl_accumulation_both_orders(zlib, cuda_device):
    """Gradient accumulation, GPT-2-XL shapes, n_dp = 4, K = 4 micro-batches:
    ZeRO-1 (fp32 local accumulation per rank, one reduce-scatter) and ZeRO-2
    (reduce-scatter per micro-batch), each against its own oracle order on
    sampled elements, then the two against each other."""
    zb = zlib
    dev = cuda_device
    n_dp, K = 4, 4
    L = zb.zero_layout(inputs.gpt2xl_numels(), n_dp, 8, 500_000_000)
    P = L.padded_n
    g = torch.empty((n_dp, P), dtype=torch.bfloat16, device=dev)
    acc = [torch.empty(P, device=dev) for _ in range(n_dp)]
    A = torch.empty(P, device=dev)
    w0 = inputs.master_weights(L.n, P, seed=SEED, device=dev)
    s1 = [w0.clone(), torch.zeros(P, device=dev), torch.zeros(P, device=dev)]
    s2 = [w0, torch.zeros(P, device=dev), torch.zeros(P, device=dev)]
    o1 = torch.zeros(P, dtype=torch.bfloat16, device=dev)
    o2 = torch.zeros(P, dtype=torch.bfloat16, device=dev)
    bounds = [b * L.bucket for b in range(1, L.n_buckets)] + [o * L.shard for o in range(1, n_dp)]
    idx = _sample_indices(0, P, bounds, seed=2)
    idx_dev = torch.from_numpy(idx).to(dev)
    w_s = parity.f32(_take(w0, idx_dev))
    samples = []
    for k in range(K):
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], L.n, SEED, step=1, rank=r, micro=k)
        samples.append(np.stack([_bits_at(g[r], idx_dev) for r in range(n_dp)]))
        zstep.zero1_accumulate_micro(L, [g[r] for r in range(n_dp)], acc, first=(k == 0))
        zstep.zero2_accumulate_micro(L, [g[r] for r in range(n_dp)], A, first=(k == 0))
    zstep.zero1_finish(L, acc, K, *s1, o1, _hp(zb, 1))
    zstep.zero2_finish(L, A, K, *s2, o2, _hp(zb, 1))
    zb.zero_status_check()
    z = np.zeros(idx.size, np.float32)
    acc_ref = [None] * n_dp
    A_ref = None
    for k, gs in enumerate(samples):
        for r in range(n_dp):
            acc_ref[r] = oracle.accumulate_local(acc_ref[r], gs[r], first=(k == 0))
        A_ref = oracle.accumulate_reduce(A_ref, gs, first=(k == 0))
    for r in range(n_dp):
        parity.assert_bit_exact_f32(_take(acc[r], idx_dev), acc_ref[r])
    parity.assert_bit_exact_f32(_take(A, idx_dev), A_ref)
    out1, *st1 = oracle.rs_adamw_reference(np.stack(acc_ref), n_dp * K, w_s, z, z, HP, 1)
    out2, *st2 = oracle.rs_adamw_reference(A_ref[None, :], n_dp * K, w_s, z, z, HP, 1)
    parity.assert_state([_take(x, idx_dev) for x in s1], st1, what="zero1 ")
    parity.assert_state([_take(x, idx_dev) for x in s2], st2, what="zero2 ")
    assert np.array_equal(_bits_at(o1, idx_dev), out1)
    assert np.array_equal(_bits_at(o2, idx_dev), out2)
    # the two orders agree within the fp32 summation bound, on every element
    x_abs = sum(np.abs(oracle.bf16_to_f32(gs).astype(np.float64)).sum(0) for gs in samples)
    bound = n_dp * K * 2.0 ** -24 / (1 - n_dp * K * 2.0 ** -24) * x_abs
    sum1 = sum(parity.f32(_take(a, idx_dev)).astype(np.float64) for a in acc)
    assert np.all(np.abs(sum1 - parity.f32(_take(A, idx_dev))) <= 2 * bound + 1e-45)
    _full_properties(s1[0], o1, L.n)
    _full_properties(s2[0], o2, L.n)


def test_llama7b_zero3_units(zlib, cuda_device):
    """ZeRO-3 per-unit path on Llama-7B units at n_dp = 8 (embedding, 32 blocks,
    head): per unit, gather the bf16 shards into one of two ring buffers for
    forward and again for backward, reduce-scatter the unit gradient into fp32,
    update the owned shards writing bf16 into each rank's own shard.  Checked on
    sampled elements of every unit; at most two units resident."""
    zb = zlib
    dev = cuda_device
    n_dp = 8
    units_numels = inputs.llama7b_units()
    layouts = [zb.zero_layout(u, n_dp) for u in units_numels]
    cap = max(L.padded_n for L in layouts)
    ring = zstep.GatherRing(cap, device=str(dev))
    gbuf = torch.empty((n_dp, cap), dtype=torch.bfloat16, device=dev)
    A = torch.empty(cap, device=dev)
    rng = np.random.default_rng(5)
    for i, L in enumerate(layouts):
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=SEED + i, device=dev)
        shards = w.to(torch.bfloat16)            # the initial bf16 shards (inputs only)
        unit = zstep.Zero3Unit(L, shards.view(n_dp, L.shard), w, torch.zeros(P, device=dev),
                               torch.zeros(P, device=dev))
        idx = np.unique(np.concatenate([rng.integers(0, P, 4096), np.arange(max(0, L.n - 8), P),
                                        [o * L.shard for o in range(n_dp)]]))
        idx_dev = torch.from_numpy(idx).to(dev)
        shard_bits = _bits_at(unit.shards.view(-1), idx_dev)
        # forward gather + release, backward gather
        buf = zstep.zero3_gather(unit, ring, ("fwd", i))
        assert np.array_equal(_bits_at(buf, idx_dev), shard_bits)
        ring.release(("fwd", i))
        buf = zstep.zero3_gather(unit, ring, ("bwd", i))
        assert torch.equal(buf.view(torch.int16), unit.shards.view(-1).view(torch.int16))
        for r in range(n_dp):
            inputs.grad_bf16_into(gbuf[r, :P], L.n, SEED, step=1, rank=r, micro=i)
        gs = np.stack([_bits_at(gbuf[r, :P], idx_dev) for r in range(n_dp)])
        ws = parity.f32(_take(w, idx_dev))
        zstep.zero3_layer_reduce_scatter(unit, [gbuf[r, :P] for r in range(n_dp)], A[:P])
        ring.release(("bwd", i))
        zstep.zero3_update(unit, A[:P], _hp(zb, 1))
        zb.zero_status_check()
        A_ref = oracle.accumulate_reduce(None, gs, first=True)
        parity.assert_bit_exact_f32(_take(A[:P], idx_dev), A_ref)
        z = np.zeros(idx.size, np.float32)
        out_ref, *st = oracle.rs_adamw_reference(A_ref[None, :], n_dp, ws, z, z, HP, 1)
        parity.assert_state([_take(x, idx_dev) for x in (unit.master, unit.m, unit.v)], st,
                            what=f"unit {i} ")
        assert np.array_equal(_bits_at(unit.shards.view(-1), idx_dev), out_ref)
        _full_properties(unit.master, unit.shards.view(-1), L.n)
        assert ring.peak <= 2
        del unit, w, shards
    assert ring.resident == 0


def test_gpt2xl_clipped_step(zlib, cuda_device):
    """GPT-2-XL shapes, n_dp = 8, 5e8-element buckets, clipping at 1.0 with
    gradients large enough that it is active.  The full-size norm is checked
    against torch (fp32 sums in rank order, an fp64 sum of squares on the
    device); updates are checked on sampled elements with the oracle, using
    the clip coefficient the oracle derives from that norm."""
    zb = zlib
    dev = cuda_device
    L = zb.zero_layout(inputs.gpt2xl_numels(), 8, 8, 500_000_000)
    P = L.padded_n
    g = torch.empty((8, P), dtype=torch.bfloat16, device=dev)
    for r in range(8):
        inputs.grad_bf16_into(g[r], L.n, SEED, step=1, rank=r, std=1e-4)
    master = inputs.master_weights(L.n, P, seed=SEED, device=dev)
    m = torch.zeros(P, device=dev)
    v = torch.zeros(P, device=dev)
    out = torch.zeros(P, dtype=torch.bfloat16, device=dev)
    bounds = [b * L.bucket for b in range(1, L.n_buckets)] + [o * L.shard for o in range(1, 8)]
    idx = _sample_indices(0, P, bounds, seed=3)
    idx_dev = torch.from_numpy(idx).to(dev)
    ws = [parity.f32(_take(x, idx_dev)) for x in (master, m, v)]
    gs = np.stack([_bits_at(g[r], idx_dev) for r in range(8)])
    bufs = zstep.NormBuffers(dev)
    zstep.zero12_step_clipped(L, [g[r] for r in range(8)], master, m, v, out, _hp(zb, 1), 1.0, bufs)
    zb.zero_status_check()
    gpu_nsq = float(bufs.norm_sq.item())
    # the norm over all 1.56e9 elements, by torch on the device
    ref_nsq = 0.0
    for lo in range(0, P, 1 << 28):
        hi = min(P, lo + (1 << 28))
        s = torch.zeros(hi - lo, dtype=torch.float32, device=dev)
        for r in range(8):
            s = s + g[r, lo:hi].float()
        gm = s / 8.0
        ref_nsq += float((gm.double() * gm.double()).sum().item())
    assert gpu_nsq == pytest.approx(ref_nsq, rel=1e-10)
    coef = oracle.clip_coef(gpu_nsq, 1.0)
    assert coef < 1.0
    ref_out, *ref = oracle.rs_adamw_reference(gs, 8, *ws, HP, 1, clip=(gpu_nsq, 1.0))
    parity.assert_state([_take(x, idx_dev) for x in (master, m, v)], ref)
    assert np.array_equal(_bits_at(out, idx_dev), ref_out)
    _full_properties(master, out, L.n)


def test_gpt2xl_int8_gradients(zlib, cuda_device):
    """GPT-2-XL shapes at n_dp = 8 with 8-bit gradients (block 256): every rank
    quantizes its whole gradient, then the fused update over all buckets,
    2 steps.  A code's scale depends on its whole block, so the oracle runs on
    sampled blocks (random ones plus those at every bucket and slice boundary
    and the ends): codes and scales of every rank, then the state and bf16
    output of every element of those blocks."""
    zb = zlib
    dev = cuda_device
    block, n_dp = 256, 8
    L = zb.zero_layout(inputs.gpt2xl_numels(), n_dp, 8, 500_000_000)
    P, S = L.padded_n, L.shard
    nb = -(-S // block)
    g = torch.empty((n_dp, P), dtype=torch.bfloat16, device=dev)
    qg = zstep.Int8Grads(L, n_dp, block, dev)
    master = inputs.master_weights(L.n, P, seed=SEED, device=dev)
    m = torch.zeros(P, device=dev)
    v = torch.zeros(P, device=dev)
    out = torch.zeros(P, dtype=torch.bfloat16, device=dev)
    # sampled blocks, as (owner, block index within the slice)
    rng = np.random.default_rng(4)
    flat = set(int(x) for x in rng.integers(0, n_dp * nb, size=2048))
    for e in [b * L.bucket for b in range(1, L.n_buckets)] + [o * S for o in range(n_dp + 1)]:
        for i in (e - 1, e):
            if 0 <= i < P:
                flat.add((i // S) * nb + (i % S) // block)
    blocks = sorted(flat)
    spans = [(o * S + j * block, o * S + min((j + 1) * block, S)) for o, j in
             (divmod(b, nb) for b in blocks)]
    idx = np.concatenate([np.arange(a, c) for a, c in spans])
    idx_dev = torch.from_numpy(idx).to(dev)
    sidx_dev = torch.tensor(blocks, device=dev)
    ref = [parity.f32(_take(x, idx_dev)) for x in (master, m, v)]
    for t in (1, 2):
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], L.n, SEED, step=t, rank=r, outlier_p=0.01)
        qg.quantize([g[r] for r in range(n_dp)])
        zstep.zero12_step_int8(L, qg, master, m, v, out, _hp(zb, t))
        zb.zero_status_check()
        gs = [_bits_at(g[r], idx_dev) for r in range(n_dp)]
        deq = np.empty((n_dp, idx.size), np.float32)
        for r in range(n_dp):
            q_got = qg.q[r].index_select(0, idx_dev).cpu().numpy()
            s_got = qg.scales[r].index_select(0, sidx_dev).cpu().numpy()
            pos = 0
            for k, (a, c) in enumerate(spans):
                q, s = oracle.quantize_int8(gs[r][pos:pos + c - a], block)
                assert np.array_equal(q_got[pos:pos + c - a], q), (t, r, a)
                assert s_got[k] == s[0], (t, r, a)
                deq[r, pos:pos + c - a] = oracle.dequantize_grad_int8(q[None, :], s[None, :], 1, block)[0]
                pos += c - a
        gm = oracle.reduce_mean(deq, n_dp)
        w2, m2, v2 = oracle.adamw(*ref, gm, HP, t)
        ref = [w2, m2, v2]
        parity.assert_state([_take(x, idx_dev) for x in (master, m, v)], ref, what=f"t={t} ")
        assert np.array_equal(_bits_at(out, idx_dev), oracle.cast_bf16(w2))
    _full_properties(master, out, L.n)


def _block_spans(S, n_dp, block, rng, n_random):
    """Sampled quantization blocks of the n_dp slices, as flat (start, end):
    random ones plus the first and last block of every slice."""
    nb = -(-S // block)
    picks = set(int(x) for x in rng.integers(0, n_dp * nb, size=n_random))
    for o in range(n_dp):
        picks.update((o * nb, o * nb + nb - 1))
    blocks = sorted(picks)
    spans = [(o * S + j * block, o * S + min((j + 1) * block, S)) for o, j in (divmod(b, nb) for b in blocks)]
    return blocks, spans


def test_llama7b_zero3_zeropp_units(zlib, cuda_device):
    """ZeRO-3 with both ZeRO++ 8-bit paths on Llama-7B units at n_dp = 8 (the
    embedding, the first and last blocks, the head), block 256: each owner
    quantizes its bf16 shard and the 8-bit gather rebuilds the unit; every rank
    quantizes its unit gradient, the owners accumulate the dequantized slices
    in fp32 and update.  Checked on sampled whole blocks of every unit: codes,
    scales, the gathered weights, the fp32 accumulation, the state and the bf16
    shards."""
    zb = zlib
    dev = cuda_device
    n_dp, block = 8, 256
    all_units = inputs.llama7b_units()
    picked = [0, 1, len(all_units) - 2, len(all_units) - 1]
    layouts = [zb.zero_layout(all_units[k], n_dp) for k in picked]
    cap = max(L.padded_n for L in layouts)
    ring = zstep.GatherRing(cap, device=str(dev))
    gbuf = torch.empty((n_dp, cap), dtype=torch.bfloat16, device=dev)
    A = torch.empty(cap, device=dev)
    rng = np.random.default_rng(6)
    for i, L in enumerate(layouts):
        P, S = L.padded_n, L.shard
        w = inputs.master_weights(L.n, P, seed=SEED + 40 + i, device=dev)
        shards = w.to(torch.bfloat16)
        unit = zstep.Zero3Unit(L, shards.view(n_dp, S), w, torch.zeros(P, device=dev),
                               torch.zeros(P, device=dev))
        blocks, spans = _block_spans(S, n_dp, block, rng, 1024)
        idx = np.concatenate([np.arange(a, c) for a, c in spans])
        idx_dev = torch.from_numpy(idx).to(dev)
        bidx_dev = torch.tensor(blocks, device=dev)
        # 8-bit weights: quantize every shard, gather
        qs = zstep.Int8Shards(L, block, dev)
        zstep.zero3_quantize(unit, qs)
        buf = zstep.zero3_gather_int8(unit, qs, ring, ("bwd", i))
        sb = _bits_at(unit.shards.view(-1), idx_dev)
        qw = qs.q.view(-1).index_select(0, idx_dev).cpu().numpy()
        sw = qs.scales[:, :qs.nb].reshape(-1).index_select(0, bidx_dev).cpu().numpy()
        gathered = _bits_at(buf, idx_dev)
        pos = 0
        for k, (a, c) in enumerate(spans):
            q, s = oracle.quantize_int8(sb[pos:pos + c - a], block)
            assert np.array_equal(qw[pos:pos + c - a], q) and sw[k] == s[0], (i, a)
            assert np.array_equal(gathered[pos:pos + c - a], oracle.dequantize_int8(q, s, block)), (i, a)
            pos += c - a
        # 8-bit gradients: quantize every rank's unit gradient, accumulate, update
        for r in range(n_dp):
            inputs.grad_bf16_into(gbuf[r, :P], L.n, SEED, step=1, rank=r, micro=i)
        qg = zstep.Int8Grads(L, n_dp, block, dev)
        qg.quantize([gbuf[r, :P] for r in range(n_dp)])
        ws = parity.f32(_take(w, idx_dev))
        zstep.zero3_layer_reduce_scatter_int8(unit, qg, A[:P])
        ring.release(("bwd", i))
        zstep.zero3_update(unit, A[:P], _hp(zb, 1))
        zb.zero_status_check()
        deq = np.empty((n_dp, idx.size), np.float32)
        for r in range(n_dp):
            g_r = _bits_at(gbuf[r, :P], idx_dev)
            q_got = qg.q[r].index_select(0, idx_dev).cpu().numpy()
            s_got = qg.scales[r].index_select(0, bidx_dev).cpu().numpy()
            pos = 0
            for k, (a, c) in enumerate(spans):
                q, s = oracle.quantize_int8(g_r[pos:pos + c - a], block)
                assert np.array_equal(q_got[pos:pos + c - a], q) and s_got[k] == s[0], (i, r, a)
                deq[r, pos:pos + c - a] = oracle.dequantize_grad_int8(q[None, :], s[None, :], 1, block)[0]
                pos += c - a
        A_ref = oracle.reduce_mean(deq, 1.0)
        parity.assert_bit_exact_f32(_take(A[:P], idx_dev), A_ref)
        z = np.zeros(idx.size, np.float32)
        out_ref, *st = oracle.rs_adamw_reference(A_ref[None, :], n_dp, ws, z, z, HP, 1)
        parity.assert_state([_take(x, idx_dev) for x in (unit.master, unit.m, unit.v)], st, what=f"unit {i} ")
        assert np.array_equal(_bits_at(unit.shards.view(-1), idx_dev), out_ref)
        _full_properties(unit.master, unit.shards.view(-1), L.n)
        del unit, w, shards, qs, qg
    assert ring.resident == 0


def test_llama7b_zero3_fused_reduce_scatter_update(zlib, cuda_device):
    """The fused per-unit reduce-scatter + update on a full Llama-7B block unit
    (202,383,360 elements, n_dp = 8), as the benchmark's fused ZeRO-3 workload
    launches it, equals the layer reduce-scatter into fp32 followed by the
    update on every element (compared on the device), two steps."""
    zb = zlib
    dev = cuda_device
    n_dp = 8
    L = zb.zero_layout(inputs.llama7b_units()[1], n_dp)
    P = L.padded_n
    w = inputs.master_weights(L.n, P, seed=SEED + 70, device=dev)
    units = [zstep.Zero3Unit(L, w.to(torch.bfloat16).view(n_dp, L.shard), w.clone(),
                             torch.zeros(P, device=dev), torch.zeros(P, device=dev)) for _ in range(2)]
    g = torch.empty((n_dp, P), dtype=torch.bfloat16, device=dev)
    A = torch.empty(P, device=dev)
    for t in (1, 2):
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], L.n, SEED, step=t, rank=r)
        rows = [g[r] for r in range(n_dp)]
        zstep.zero3_layer_reduce_scatter(units[0], rows, A)
        zstep.zero3_update(units[0], A, _hp(zb, t))
        zstep.zero3_reduce_scatter_update(units[1], rows, _hp(zb, t))
        zb.zero_status_check()
        for a, b in ((units[0].master, units[1].master), (units[0].m, units[1].m), (units[0].v, units[1].v)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert torch.equal(units[0].shards.view(torch.int16), units[1].shards.view(torch.int16))
    _full_properties(units[1].master, units[1].shards.view(-1), L.n)


def test_llama7b_zero3_fused_q8_update(zlib, cuda_device):
    """The fused reduce-scatter + update with the 8-bit output on a full Llama-7B
    block unit laid out with align 256 (n_dp = 8), as the benchmark's fused
    8-bit ZeRO-3 workload launches it, equals the reduce-scatter into fp32, the
    update into bf16 shards and the quantizer, on every element and scale
    (compared on the device), two steps."""
    zb = zlib
    dev = cuda_device
    n_dp = 8
    L = zb.zero_layout(inputs.llama7b_units()[1], n_dp, align=256)
    P = L.padded_n
    w = inputs.master_weights(L.n, P, seed=SEED + 80, device=dev)
    units = [zstep.Zero3Unit(L, w.to(torch.bfloat16).view(n_dp, L.shard), w.clone(),
                             torch.zeros(P, device=dev), torch.zeros(P, device=dev)) for _ in range(2)]
    qs = [zstep.Int8Shards(L, 256, dev) for _ in range(2)]
    g = torch.empty((n_dp, P), dtype=torch.bfloat16, device=dev)
    A = torch.empty(P, device=dev)
    for t in (1, 2):
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], L.n, SEED, step=t, rank=r)
        rows = [g[r] for r in range(n_dp)]
        zstep.zero3_layer_reduce_scatter(units[0], rows, A)
        zstep.zero3_update(units[0], A, _hp(zb, t))
        zstep.zero3_quantize(units[0], qs[0])
        zstep.zero3_reduce_scatter_update_q8(units[1], rows, qs[1], _hp(zb, t))
        zb.zero_status_check()
        for a, b in ((units[0].master, units[1].master), (units[0].m, units[1].m), (units[0].v, units[1].v)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert torch.equal(qs[0].q, qs[1].q)
        assert torch.equal(qs[0].scales.view(torch.int32), qs[1].scales.view(torch.int32))


def test_llama7b_zero3_fused_int8_gradients_q8(zlib, cuda_device):
    """Both ZeRO++ 8-bit paths fused on a full Llama-7B block unit laid out with
    align 256 (n_dp = 8), as the benchmark's fused ZeRO++ workload launches it:
    from the ranks' 8-bit gradients straight to 8-bit shards, equal on every
    element and scale to the 8-bit accumulation into fp32, the update into bf16
    and the quantizer (compared on the device), two steps."""
    zb = zlib
    dev = cuda_device
    n_dp = 8
    L = zb.zero_layout(inputs.llama7b_units()[1], n_dp, align=256)
    P = L.padded_n
    w = inputs.master_weights(L.n, P, seed=SEED + 90, device=dev)
    units = [zstep.Zero3Unit(L, w.to(torch.bfloat16).view(n_dp, L.shard), w.clone(),
                             torch.zeros(P, device=dev), torch.zeros(P, device=dev)) for _ in range(2)]
    qs = [zstep.Int8Shards(L, 256, dev) for _ in range(2)]
    qg = zstep.Int8Grads(L, n_dp, 256, dev)
    g = torch.empty((n_dp, P), dtype=torch.bfloat16, device=dev)
    A = torch.empty(P, device=dev)
    for t in (1, 2):
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], L.n, SEED, step=t, rank=r, outlier_p=0.01)
        qg.quantize([g[r] for r in range(n_dp)])
        zstep.zero3_layer_reduce_scatter_int8(units[0], qg, A)
        zstep.zero3_update(units[0], A, _hp(zb, t))
        zstep.zero3_quantize(units[0], qs[0])
        zstep.zero3_reduce_scatter_update_int8_q8(units[1], qg, qs[1], _hp(zb, t))
        zb.zero_status_check()
        for a, b in ((units[0].master, units[1].master), (units[0].m, units[1].m), (units[0].v, units[1].v)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert torch.equal(qs[0].q, qs[1].q)
        assert torch.equal(qs[0].scales.view(torch.int32), qs[1].scales.view(torch.int32))


def test_llama7b_zero3_fused_graph_replay(zlib, cuda_device):
    """The fused ZeRO-3 step captured once in a CUDA graph, as the benchmark's
    graph workload captures it (the schedule's advance, then per unit the
    forward gather, and in reverse the backward gather with the fused
    reduce-scatter + update), on the Llama-7B embedding and two block units at
    n_dp = 8.  The capture's warm-up call is step 1; three replays with new
    gradients in the same buffer and a new lr each step equal four eager steps
    with the scalars by value on every element, and the oracle on sampled
    elements."""
    zb = zlib
    dev = cuda_device
    n_dp = 8
    units_numels = inputs.llama7b_units()[:3]
    layouts = [zb.zero_layout(u, n_dp) for u in units_numels]
    cap = max(L.padded_n for L in layouts)
    lrs = [1e-4, 8e-5, 6e-5, 4e-5]

    def make_units(seed):
        out = []
        for i, L in enumerate(layouts):
            w = inputs.master_weights(L.n, L.padded_n, seed=seed + i, device=dev)
            out.append(zstep.Zero3Unit(L, w.to(torch.bfloat16).view(n_dp, L.shard), w,
                                       torch.zeros(L.padded_n, device=dev), torch.zeros(L.padded_n, device=dev)))
        return out

    def step_ops(units, ring, gbuf, hp_of):
        for i, u in enumerate(units):
            zstep.zero3_gather(u, ring, ("fwd", i))
            ring.release(("fwd", i))
        for i in reversed(range(len(units))):
            u = units[i]
            P = u.layout.padded_n
            zstep.zero3_gather(u, ring, ("bwd", i))
            zstep.zero3_reduce_scatter_update(u, [gbuf[r, :P] for r in range(n_dp)], hp_of())
            ring.release(("bwd", i))

    def fill(gbuf, t):
        for r in range(n_dp):
            inputs.grad_bf16_into(gbuf[r], cap, SEED + 90, step=t, rank=r)

    graph_units, eager_units = make_units(SEED + 80), make_units(SEED + 80)
    u0 = graph_units[0]
    rng = np.random.default_rng(9)
    idx = np.unique(np.concatenate([rng.integers(0, u0.layout.padded_n, 1 << 16),
                                    [o * u0.layout.shard for o in range(n_dp)]]))
    idx_dev = torch.from_numpy(idx).to(dev)
    ref = [parity.f32(_take(u0.master, idx_dev)), np.zeros(idx.size, np.float32),
           np.zeros(idx.size, np.float32)]

    gbuf = torch.empty((n_dp, cap), dtype=torch.bfloat16, device=dev)      # the graph's fixed input
    ring = zstep.GatherRing(cap, device=str(dev))
    sch = zstep.StepSchedule(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, n_steps=len(lrs), lrs=lrs)

    def graph_step():
        sch.advance()
        step_ops(graph_units, ring, gbuf, sch.hp)

    fill(gbuf, 1)
    gs = zstep.GraphStep(graph_step)                                       # warm-up = step 1
    for t in range(2, len(lrs) + 1):
        fill(gbuf, t)
        gs.replay()
    torch.cuda.synchronize()
    assert int(sch.index.item()) == len(lrs)

    ebuf = torch.empty_like(gbuf)
    ering = zstep.GatherRing(cap, device=str(dev))
    o = oracle.AdamW(lr=HP.lr, beta1=HP.beta1, beta2=HP.beta2, eps=HP.eps, weight_decay=HP.weight_decay)
    for t in range(1, len(lrs) + 1):
        fill(ebuf, t)
        hp = zb.ZeroAdamW.make(lrs[t - 1], HP.beta1, HP.beta2, HP.eps, HP.weight_decay, t)
        step_ops(eager_units, ering, ebuf, lambda: hp)
        gs_bits = np.stack([_bits_at(ebuf[r, :u0.layout.padded_n], idx_dev) for r in range(n_dp)])
        o.lr = float(np.float32(lrs[t - 1]))
        out_ref, *ref = oracle.rs_adamw_reference(gs_bits, n_dp, *ref, o, t)
    zb.zero_status_check()
    for g_u, e_u in zip(graph_units, eager_units):
        for a, b in ((g_u.master, e_u.master), (g_u.m, e_u.m), (g_u.v, e_u.v)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert torch.equal(g_u.shards.view(torch.int16), e_u.shards.view(torch.int16))
    parity.assert_state([_take(x, idx_dev) for x in (u0.master, u0.m, u0.v)], ref, what="graph unit 0 ")
    assert np.array_equal(_bits_at(u0.shards.view(-1), idx_dev), out_ref)
    assert ring.resident == 0 and ering.resident == 0
