"""Per-step scalars in device memory and steps captured in CUDA graphs.

The update kernels can read lr and the bias corrections of the current step
from device memory (zero_adamw_t::sched), written by zero_schedule_advance
from a table that zero_schedule_fill computes on the host exactly as for a
by-value step.  So: every kind of update gives bit-identical results either
way, and a step captured once in a CUDA graph, then replayed, equals the
eager steps one after another -- with a per-step learning rate too."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

LR, B1, B2, EPS, WD = 3e-4, 0.9, 0.95, 1e-8, 0.1


def _by_value(zb, t, lr=LR):
    return zb.ZeroAdamW.make(lr, B1, B2, EPS, WD, t)


def _state(N, P, seed):
    w = inputs.master_weights(N, P, seed=seed).cuda()
    return [w, torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]


def _equal(a, b):
    for x, y in zip(a, b):
        parity.assert_bit_exact_f32(x, parity.f32(y))


@pytest.mark.parametrize("kind", ["bf16", "f32", "q8", "int8", "int8_q8", "clip"])
def test_device_scalars_equal_by_value_scalars(zlib, cuda_device, kind):
    zb = zlib
    n_dp, N = 4, 100_003
    L = zb.zero_layout([N], n_dp, align=256, bucket_elems=30_000)
    P = L.padded_n
    sch = zstep.StepSchedule(LR, B1, B2, EPS, WD, n_steps=3, lrs=[1e-3, 3e-4, 5e-5])
    a, b = _state(N, P, 1), _state(N, P, 1)
    oa = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    ob = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    qa = [torch.zeros(P, dtype=torch.int8, device="cuda"), torch.zeros(P // 256, device="cuda")]
    qb = [torch.zeros(P, dtype=torch.int8, device="cuda"), torch.zeros(P // 256, device="cuda")]
    for t, lr in zip((1, 2, 3), (1e-3, 3e-4, 5e-5)):
        sch.advance()
        g = inputs.grads_bf16(n_dp, N, P, seed=2, step=t, std=1.0 if kind == "clip" else 1e-3)
        gd = [g[r].cuda() for r in range(n_dp)]
        hv, hd = _by_value(zb, t, lr), sch.hp()
        if kind == "bf16":
            zstep.zero12_step(L, gd, *a, oa, hv)
            zstep.zero12_step(L, gd, *b, ob, hd)
        elif kind == "f32":
            A = torch.stack(gd).float().sum(0)
            zb.zero_reduce_scatter_adamw(L, [A], zb.ZERO_F32, 0, float(n_dp), 0, n_dp, 0, P, *a, oa,
                                         zb.ZERO_OUT_SHARD, hv)
            zb.zero_reduce_scatter_adamw(L, [A], zb.ZERO_F32, 0, float(n_dp), 0, n_dp, 0, P, *b, ob,
                                         zb.ZERO_OUT_SHARD, hd)
        elif kind == "q8":
            zb.zero_reduce_scatter_adamw_q8(L, gd, zb.ZERO_BF16, 0, float(n_dp), 0, n_dp, 0, P, *a, *qa, 256, hv)
            zb.zero_reduce_scatter_adamw_q8(L, gd, zb.ZERO_BF16, 0, float(n_dp), 0, n_dp, 0, P, *b, *qb, 256, hd)
        elif kind in ("int8", "int8_q8"):
            qg = zstep.Int8Grads(L, n_dp, 256)
            qg.quantize(gd)
            q, s = qg.sources()
            if kind == "int8":
                for hp, st, o in ((hv, a, oa), (hd, b, ob)):
                    zb.zero_reduce_scatter_adamw_int8(L, q, s, 256, float(n_dp), 0, n_dp, 0, P, *st, o,
                                                      zb.ZERO_OUT_FULL, hp)
            else:
                zb.zero_reduce_scatter_adamw_int8_q8(L, q, s, 256, float(n_dp), 0, n_dp, 0, P, *a, *qa, 256, hv)
                zb.zero_reduce_scatter_adamw_int8_q8(L, q, s, 256, float(n_dp), 0, n_dp, 0, P, *b, *qb, 256, hd)
        else:
            bufs = zstep.NormBuffers("cuda")
            zstep.zero12_step_clipped(L, gd, *a, oa, hv, 1.0, bufs)
            zstep.zero12_step_clipped(L, gd, *b, ob, hd, 1.0, bufs)
        torch.cuda.synchronize()
        _equal(a, b)
        assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
        assert torch.equal(qa[0], qb[0]) and torch.equal(qa[1], qb[1])
    zb.zero_status_check()


def test_graph_replays_equal_eager_steps(zlib, cuda_device):
    """A ZeRO-2 step (schedule advance + the bucketed fused update) captured once
    and replayed 3 times equals 4 eager steps (the capture's warm-up call is a
    real step), with a different lr per step; the oracle agrees."""
    zb = zlib
    n_dp, N = 8, 300_007
    L = zb.zero_layout([N], n_dp, bucket_elems=100_000)
    P = L.padded_n
    lrs = [1e-3, 5e-4, 2e-4, 1e-4]
    eager, graph = _state(N, P, 3), _state(N, P, 3)
    w0 = parity.f32(eager[0])
    oe = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    og = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    gbuf = torch.empty((n_dp, P), dtype=torch.bfloat16, device="cuda")      # the graph's fixed input
    rows = [gbuf[r] for r in range(n_dp)]
    sch = zstep.StepSchedule(LR, B1, B2, EPS, WD, n_steps=len(lrs), lrs=lrs)

    def step():
        sch.advance()
        zstep.zero12_step(L, rows, *graph, og, sch.hp())

    grads = [inputs.grads_bf16(n_dp, N, P, seed=4, step=t) for t in range(1, 5)]
    gbuf.copy_(grads[0])
    gs = zstep.GraphStep(step)                                  # warm-up = step 1
    for t in range(2, 5):
        gbuf.copy_(grads[t - 1])
        gs.replay()
    ref = [w0, np.zeros(P, np.float32), np.zeros(P, np.float32)]
    o = oracle.AdamW(lr=LR, beta1=B1, beta2=B2, eps=EPS, weight_decay=WD)
    for t in range(1, 5):
        zstep.zero12_step(L, [grads[t - 1][r].cuda() for r in range(n_dp)], *eager, oe,
                          _by_value(zb, t, lrs[t - 1]))
        o.lr = float(np.float32(lrs[t - 1]))
        out_ref, *ref = oracle.rs_adamw_reference(parity.bits(grads[t - 1]), n_dp, *ref, o, t)
    torch.cuda.synchronize()
    _equal(graph, eager)
    assert torch.equal(og.view(torch.int16), oe.view(torch.int16))
    parity.assert_state(graph, ref)
    assert np.array_equal(parity.bits(og), out_ref)
    assert int(sch.index.item()) == 4
    zb.zero_status_check()


def test_schedule_past_its_table_is_reported(zlib, cuda_device):
    zb = zlib
    sch = zstep.StepSchedule(LR, B1, B2, EPS, WD, n_steps=2)
    sch.advance()
    sch.advance()
    zb.zero_status_check()
    sch.advance()                                               # index 2 of a 2-row table
    with pytest.raises(zb.ZeroError) as e:
        zb.zero_status_check()
    assert e.value.code == zb.ZERO_ERANGE
    assert int(sch.index.item()) == 2
    zb.zero_status_check()                                      # reported once


def test_the_adamw_block_keeps_its_schedule_memory(zlib, cuda_device):
    """A block made with sched=<a temporary tensor> holds that tensor, so the
    pointer it carries stays valid after the caller drops its own reference."""
    import gc
    import weakref
    zb = zlib
    hp = zb.ZeroAdamW.make(LR, B1, B2, EPS, WD, 1, sched=torch.tensor([LR, 0.1, 0.001], device="cuda"))
    ref = weakref.ref(hp._sched_tensor)
    gc.collect()
    assert ref() is not None and hp.sched == ref().data_ptr()
    del hp
    gc.collect()
    assert ref() is None
