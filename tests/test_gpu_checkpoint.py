"""Checkpoint and resume on the GPU, against the oracle ("ZeRO Optimizer, in
depth", "Checkpoints: sharded on the way in, consolidated on the way out").

A run saved after two steps is checked three ways: the consolidated state
(every rank's shard concatenated, padding dropped) equals the oracle's state
after the same two steps; restored into fresh device buffers and continued, it
ends where the oracle's steps from the saved state end and where the same run
without the interruption ends; resharded to another rank count, it restores
element for element and a step at the new count gives the oracle's step at
that count.  The stage-3 unit checkpoints get the same checks."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import checkpoint as ck
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

HP = oracle.AdamW()        # the hyper-parameters of ZeroAdamW.make's defaults


def _grads(L, t):
    return inputs.grads_bf16(L.n_dp, L.n, L.padded_n, seed=8, step=t)


def _run(zb, L, state, out, t0, t1):
    for t in range(t0, t1):
        g = _grads(L, t)
        zstep.zero12_step(L, [g[r].cuda() for r in range(L.n_dp)], *state, out,
                          zb.ZeroAdamW.make(step=t))


def _oracle_run(L, w, m, v, t0, t1):
    """oracle.zero_step for steps t0..t1-1 from flat padded fp32 state."""
    n_dp, S = L.n_dp, L.shard
    w, m, v = (np.asarray(x, np.float32).reshape(n_dp, S) for x in (w, m, v))
    full = None
    for t in range(t0, t1):
        full, w, m, v = oracle.zero_step(parity.bits(_grads(L, t)), w, m, v, HP, t)
    return full[0], w.reshape(-1), m.reshape(-1), v.reshape(-1)


def test_save_restore_continue(zlib, cuda_device, tmp_path):
    zb = zlib
    numels = [300_000, 17, 99_999]
    L = zb.zero_layout(numels, 4, bucket_elems=100_000)
    P, N = L.padded_n, L.n
    w0 = inputs.master_weights(N, P, seed=8).cuda()
    zeros = np.zeros(P, np.float32)
    ref = [w0.clone(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    ref_out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    _run(zb, L, ref, ref_out, 1, 5)
    st = [w0.clone(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    _run(zb, L, st, out, 1, 3)
    ck.save(str(tmp_path / "c"), L, numels, *st, 2, zb.ZeroAdamW.make(step=2), out_bf16=out)
    # the consolidated state is the oracle's after two steps, padding dropped
    o_full2, *o_st2 = _oracle_run(L, parity.f32(w0), zeros, zeros, 1, 3)
    flat = ck.consolidate(str(tmp_path / "c"))
    assert flat["step"] == 2 and all(flat[k].size == N for k in ("master", "m", "v"))
    parity.assert_state([flat["master"], flat["m"], flat["v"]], [x[:N] for x in o_st2], what="consolidated ")
    per = ck.consolidate(str(tmp_path / "c"), split=True)["tensors"]
    offs = np.cumsum([0] + numels[:-1])
    for k, (off, cnt) in enumerate(zip(offs, numels)):
        np.testing.assert_array_equal(per[k]["master"], flat["master"][off:off + cnt])
    assert np.array_equal(parity.bits(out), o_full2)
    # restored into fresh buffers and continued: the oracle's steps 3 and 4 from
    # the saved state, and the run without the interruption
    fresh = [torch.full((P,), float("nan"), device="cuda") for _ in range(3)]
    fresh_out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    t = ck.restore(str(tmp_path / "c"), L, *fresh, out_bf16=fresh_out)
    assert t == 2
    assert torch.equal(fresh_out.view(torch.int16), out.view(torch.int16))
    _run(zb, L, fresh, fresh_out, t + 1, 5)
    torch.cuda.synchronize()
    saved = [np.concatenate([flat[k], np.zeros(P - N, np.float32)]) for k in ("master", "m", "v")]
    o_full4, *o_st4 = _oracle_run(L, *saved, t + 1, 5)
    parity.assert_state(fresh, o_st4, what="resumed ")
    assert np.array_equal(parity.bits(fresh_out), o_full4)
    for a, b in zip(fresh, ref):
        parity.assert_bit_exact_f32(a, b)
    assert torch.equal(fresh_out.view(torch.int16), ref_out.view(torch.int16))
    # resharded to 3 ranks: the state restores into the 3-rank layout element
    # for element, and a step at 3 ranks is the oracle's step at 3 ranks
    ck.reshard(str(tmp_path / "c"), str(tmp_path / "d"), 3)
    L3 = zb.zero_layout(numels, 3, bucket_elems=100_000)
    st3 = [torch.zeros(L3.padded_n, device="cuda") for _ in range(3)]
    assert ck.restore(str(tmp_path / "d"), L3, *st3) == 2
    for a3, a in zip(st3, st):
        np.testing.assert_array_equal(parity.f32(a3)[:N], parity.f32(a)[:N])
        assert not parity.f32(a3)[N:].any()
    start3 = [parity.f32(x).copy() for x in st3]
    out3 = torch.zeros(L3.padded_n, dtype=torch.bfloat16, device="cuda")
    _run(zb, L3, st3, out3, 3, 4)
    torch.cuda.synchronize()
    o_full3, *o_st3 = _oracle_run(L3, *start3, 3, 4)
    parity.assert_state(st3, o_st3, what="resharded ")
    assert np.array_equal(parity.bits(out3), o_full3)


def _units(zb, numels_list, n_dp):
    units = []
    for i, numels in enumerate(numels_list):
        L = zb.zero_layout(numels, n_dp)
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=90 + i).cuda()
        shards = torch.empty(P, dtype=torch.bfloat16, device="cuda")
        zb.zero_cast_bf16(w, shards)
        units.append(zstep.Zero3Unit(L, shards.view(n_dp, L.shard), w,
                                     torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")))
    return units


def _unit_grads(L, i, t):
    return inputs.grads_bf16(L.n_dp, L.n, L.padded_n, seed=95 + i, step=t)


def _units_step(zb, units, t):
    cap = max(u.layout.padded_n for u in units)
    A = torch.empty(cap, device="cuda")
    for i in reversed(range(len(units))):
        u = units[i]
        P = u.layout.padded_n
        g = _unit_grads(u.layout, i, t)
        zstep.zero3_layer_reduce_scatter(u, [g[r].cuda() for r in range(u.layout.n_dp)], A[:P])
        zstep.zero3_update(u, A[:P], zb.ZeroAdamW.make(step=t))


def _oracle_units(layouts, states, shards, t0, t1):
    _, st, sh = parity.zero3_oracle_run(
        states, shards,
        [lambda t, i=i, L=L: parity.bits(_unit_grads(L, i, t)) for i, L in enumerate(layouts)],
        HP, range(t0, t1), layouts[0].n_dp)
    return st, sh


def test_stage3_unit_checkpoints(zlib, cuda_device, tmp_path):
    zb = zlib
    n_dp = 4
    numels_list = [[4097], [1000, 24, 3, 5000], [7]]
    units = _units(zb, numels_list, n_dp)
    layouts = [u.layout for u in units]
    init = [[parity.f32(u.master), np.zeros(u.layout.padded_n, np.float32),
             np.zeros(u.layout.padded_n, np.float32)] for u in units]
    init_sh = [parity.bits(u.shards).reshape(-1) for u in units]
    for t in (1, 2):
        _units_step(zb, units, t)
    ck.save_units(str(tmp_path / "u"), units, numels_list, 2, zb.ZeroAdamW.make(step=2), with_bf16=True)
    st2, sh2 = _oracle_units(layouts, init, init_sh, 1, 3)
    # consolidated: every unit's real elements, units in order
    flat = ck.consolidate_units(str(tmp_path / "u"))
    for k, key in enumerate(("master", "m", "v")):
        ref = np.concatenate([st2[i][k][:L.n] for i, L in enumerate(layouts)])
        parity.assert_f32_close(flat[key], ref, what=f"consolidated {key}")
    # restored into fresh units and continued one step: the oracle's step 3
    fresh = _units(zb, numels_list, n_dp)
    for u in fresh:
        for x in (u.master, u.m, u.v):
            x.fill_(float("nan"))
        u.shards.zero_()
    assert ck.restore_units(str(tmp_path / "u"), fresh, with_bf16=True) == 2
    for i, u in enumerate(fresh):
        assert np.array_equal(parity.bits(u.shards).reshape(-1), sh2[i])
    _units_step(zb, fresh, 3)
    torch.cuda.synchronize()
    st3, sh3 = _oracle_units(layouts, st2, sh2, 3, 4)
    for i, u in enumerate(fresh):
        parity.assert_state([u.master, u.m, u.v], st3[i], what=f"unit {i} ")
        assert np.array_equal(parity.bits(u.shards).reshape(-1), sh3[i])
    # resharded to 3 ranks: every unit's real elements restore unchanged
    ck.reshard_units(str(tmp_path / "u"), str(tmp_path / "u3"), 3)
    units3 = _units(zb, numels_list, 3)
    assert ck.restore_units(str(tmp_path / "u3"), units3) == 2
    for i, (u3, L) in enumerate(zip(units3, layouts)):
        for k, x in enumerate((u3.master, u3.m, u3.v)):
            np.testing.assert_array_equal(parity.f32(x)[:L.n], st2[i][k][:L.n])
            assert not parity.f32(x)[L.n:].any()
