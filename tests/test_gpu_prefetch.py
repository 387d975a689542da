"""ZeRO-3 with gathers one unit ahead on a side stream ("ZeRO and FSDP",
"FSDP, ZeRO-3 inside PyTorch": the next unit is gathered while the current one
computes, at most two resident): every gathered unit and the final state equal
the oracle's stage-3 sequence, and the sequential path, bit for bit."""
import numpy as np
import pytest
import torch

import oracle

from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu


def _units(zb, numels_list, n_dp, seed):
    units = []
    for i, numels in enumerate(numels_list):
        L = zb.zero_layout(numels, n_dp)
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=seed + i).cuda()
        shards = torch.empty(P, dtype=torch.bfloat16, device="cuda")
        zb.zero_cast_bf16(w, shards)
        units.append(zstep.Zero3Unit(L, shards.view(n_dp, L.shard), w,
                                     torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")))
    return units


@pytest.mark.parametrize("int8", [False, True])
def test_prefetched_equals_sequential(zlib, cuda_device, int8):
    zb = zlib
    n_dp = 8
    numels_list = [[131_072], [200_000, 8], [7], [65_536, 4097], [262_144]]
    a = _units(zb, numels_list, n_dp, 60)
    b = _units(zb, numels_list, n_dp, 60)
    cap = max(u.layout.padded_n for u in a)
    grads = [inputs.grads_bf16(n_dp, u.layout.n, u.layout.padded_n, seed=70 + i, step=1).cuda()
             for i, u in enumerate(a)]
    qa = [zstep.Int8Shards(u.layout, 256) for u in a] if int8 else None
    qb = [zstep.Int8Shards(u.layout, 256) for u in b] if int8 else None
    if int8:
        for u, q in zip(a, qa):
            zstep.zero3_quantize(u, q)
        for u, q in zip(b, qb):
            zstep.zero3_quantize(u, q)
    seen = {"a": [], "b": []}

    def compute(which):
        def f(i, buf, phase):
            seen[which].append((phase, i, buf.clone()))
        return f

    ring_a = zstep.GatherRing(cap)
    A = torch.empty(cap, device="cuda")
    pf = zstep.Zero3Prefetcher(a, ring_a, int8=qa)
    for t in (1, 2):
        zstep.zero3_step_prefetched(pf, lambda i: [grads[i][r] for r in range(n_dp)], A,
                                    zb.ZeroAdamW.make(step=t), compute("a"))
    # the sequential reference
    ring_b = zstep.GatherRing(cap)
    B = torch.empty(cap, device="cuda")
    for t in (1, 2):
        for i, u in enumerate(b):
            buf = (zstep.zero3_gather_int8(u, qb[i], ring_b, "f") if int8 else
                   zstep.zero3_gather(u, ring_b, "f"))
            seen["b"].append(("fwd", i, buf.clone()))
            ring_b.release("f")
        for i in reversed(range(len(b))):
            u = b[i]
            P = u.layout.padded_n
            buf = (zstep.zero3_gather_int8(u, qb[i], ring_b, "b") if int8 else
                   zstep.zero3_gather(u, ring_b, "b"))
            seen["b"].append(("bwd", i, buf.clone()))
            zstep.zero3_layer_reduce_scatter(u, [grads[i][r] for r in range(n_dp)], B[:P])
            ring_b.release("b")
            zstep.zero3_update(u, B[:P], zb.ZeroAdamW.make(step=t))
            if int8:
                zstep.zero3_quantize(u, qb[i])
    torch.cuda.synchronize()
    assert ring_a.peak <= 2 and ring_a.resident == 0
    assert [(p, i) for p, i, _ in seen["a"]] == [(p, i) for p, i, _ in seen["b"]]
    for (_, _, x), (_, _, y) in zip(seen["a"], seen["b"]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for ua, ub in zip(a, b):
        for x, y in ((ua.master, ub.master), (ua.m, ub.m), (ua.v, ub.v)):
            parity.assert_bit_exact_f32(x, y)
        assert torch.equal(ua.shards.view(torch.int16), ub.shards.view(torch.int16))
    # the oracle's sequence from the same initial state: every gathered unit at
    # the moment it was gathered, and the final master / m / v / shards
    init = _units(zb, numels_list, n_dp, 60)
    host_grads = [parity.bits(g) for g in grads]
    gathered, st, sh = parity.zero3_oracle_run(
        [[parity.f32(u.master), np.zeros(u.layout.padded_n, np.float32), np.zeros(u.layout.padded_n, np.float32)]
         for u in init],
        [parity.bits(u.shards).reshape(-1) for u in init],
        [lambda t, g=g: g for g in host_grads], oracle.AdamW(), (1, 2), n_dp, 256 if int8 else None)
    assert [(p, i) for p, i, _ in seen["a"]] == [(p, i) for p, i, _ in gathered]
    for (p, i, x), (_, _, ref) in zip(seen["a"], gathered):
        assert np.array_equal(parity.bits(x), ref), (p, i)
    for i, ua in enumerate(a):
        parity.assert_state([ua.master, ua.m, ua.v], st[i], what=f"unit {i} ")
        assert np.array_equal(parity.bits(ua.shards).reshape(-1), sh[i])
