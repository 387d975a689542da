"""The configuration-driven engines against the oracle: every branch the
engines choose (fused, accumulating, clipped, 8-bit) gives the oracle's step."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep
from zero_sharded_mixed_gb300.config import ZeroConfig
from zero_sharded_mixed_gb300.engine import Zero3Engine, ZeroEngine

pytestmark = pytest.mark.gpu

HP = oracle.AdamW(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def _cfg(**kw):
    base = {"gradient_accumulation_steps": kw.pop("K", 1), "gradient_clipping": kw.pop("clip", 0.0),
            "optimizer": {"type": "AdamW", "params": {"lr": HP.lr, "betas": [HP.beta1, HP.beta2],
                                                      "eps": HP.eps, "weight_decay": HP.weight_decay}},
            "zero_optimization": {"stage": kw.pop("stage"), "reduce_bucket_size": kw.pop("bucket", 30_000),
                                  "zero_quantized_weights": kw.pop("qw", False),
                                  "zero_quantized_gradients": kw.pop("qg", False)}}
    assert not kw
    return ZeroConfig.from_dict(base)


def _oracle_step(rows_per_micro, n_dp, state, t, clip, qg, stage):
    """The oracle's step for K micro-batches of bf16 rows: the accumulation
    order of the stage, the optional 8-bit gradients, clipping, the update."""
    K = len(rows_per_micro)
    if qg:
        A = None
        for k, rows in enumerate(rows_per_micro):
            q, s = oracle.quantize_grad_int8(rows, n_dp, 256)
            A = oracle.accumulate_reduce_int8(A, q, s, n_dp, 256, k == 0)
        src = A[None, :]
    elif stage == 1:
        acc = [None] * n_dp
        for k, rows in enumerate(rows_per_micro):
            acc = [oracle.accumulate_local(acc[r], rows[r], k == 0) for r in range(n_dp)]
        src = np.stack(acc)
    else:
        A = None
        for k, rows in enumerate(rows_per_micro):
            A = oracle.accumulate_reduce(A, rows, k == 0)
        src = A[None, :]
    if K == 1 and not qg:
        src = rows_per_micro[0]
    clip_arg = None
    if clip:
        clip_arg = (oracle.grad_norm_sq(src, n_dp * K), clip)
    return oracle.rs_adamw_reference(src, n_dp * K, *state, HP, t, clip=clip_arg)


@pytest.mark.parametrize("stage,K,clip,qg", [
    (2, 1, 0.0, False), (1, 3, 0.0, False), (2, 3, 0.0, False), (1, 1, 1.0, False),
    (2, 3, 1.0, False), (1, 3, 1.0, False), (2, 1, 0.0, True), (2, 2, 0.0, True), (1, 1, 0.5, True),
])
def test_zero12_engine(zlib, cuda_device, stage, K, clip, qg):
    n_dp, N = 4, 100_003
    eng = ZeroEngine([N], n_dp, _cfg(stage=stage, K=K, clip=clip, qg=qg),
                     master=inputs.master_weights(N, 100_032, seed=1).cuda())
    P = eng.L.padded_n
    state = [parity.f32(eng.master), np.zeros(P, np.float32), np.zeros(P, np.float32)]
    std = 1.0 if clip else 1e-3
    for t in (1, 2):
        micro = []
        for k in range(K):
            g = inputs.grads_bf16(n_dp, N, P, seed=t, step=t, micro=k, std=std)
            micro.append(parity.bits(g))
            eng.backward(g.cuda())
        eng.step()
        torch.cuda.synchronize()
        out_ref, *state = _oracle_step(micro, n_dp, state, t, clip, qg, stage)
        parity.assert_state([eng.master, eng.m, eng.v], state, exact=not clip, what=f"t={t} ")
        if clip:
            parity.assert_bf16_close(eng.weights, out_ref)
        else:
            assert np.array_equal(parity.bits(eng.weights), out_ref)
    with pytest.raises(RuntimeError):
        eng.step()                                           # no micro-batch given


@pytest.mark.parametrize("K,clip,qw,qg", [
    (1, 0.0, False, False), (1, 0.0, True, False), (1, 0.0, False, True), (1, 0.0, True, True),
    (2, 0.0, False, False), (2, 0.0, True, True), (1, 1.0, True, False), (2, 1.0, False, False),
])
def test_zero3_engine(zlib, cuda_device, K, clip, qw, qg):
    n_dp = 5
    units = [[4097], [33_031], [1000, 24, 3, 5000]]
    eng = Zero3Engine(units, n_dp, _cfg(stage=3, K=K, clip=clip, qw=qw, qg=qg))
    for i, u in enumerate(eng.units):                        # start from seeded weights
        u.master.copy_(inputs.master_weights(u.layout.n, u.layout.padded_n, seed=10 + i).cuda())
    std = 1.0 if clip else 1e-3
    states = [[parity.f32(u.master), np.zeros(u.layout.padded_n, np.float32),
               np.zeros(u.layout.padded_n, np.float32)] for u in eng.units]
    micro_rows = [[] for _ in eng.units]
    for k in range(K):
        for i in reversed(range(len(eng.units))):            # backward order
            u = eng.units[i]
            buf = eng.gather(i)
            assert buf.numel() == u.layout.padded_n
            eng.release(i)
            g = inputs.grads_bf16(n_dp, u.layout.n, u.layout.padded_n, seed=20 + i, step=1, micro=k, std=std)
            micro_rows[i].append(parity.bits(g))
            eng.backward(i, g.cuda(), micro=k)
    eng.step()
    torch.cuda.synchronize()
    # the oracle: per unit the reduced gradient, the global norm over all units, the update
    srcs = []
    for i in range(len(eng.units)):
        if qg:
            A = None
            for k, rows in enumerate(micro_rows[i]):
                q, s = oracle.quantize_grad_int8(rows, n_dp, 256)
                A = oracle.accumulate_reduce_int8(A, q, s, n_dp, 256, k == 0)
        else:
            A = None
            for k, rows in enumerate(micro_rows[i]):
                A = oracle.accumulate_reduce(A, rows, k == 0)
        srcs.append(A[None, :])
    clip_arg = None
    if clip:
        clip_arg = (sum(oracle.grad_norm_sq(s, n_dp * K) for s in srcs), clip)
    for i, u in enumerate(eng.units):
        out_ref, *st = oracle.rs_adamw_reference(srcs[i], n_dp * K, *states[i], HP, 1, clip=clip_arg)
        parity.assert_state([u.master, u.m, u.v], st, what=f"unit {i} ")
        S = u.layout.shard
        if qw:
            q = eng.q8[i]
            for o in range(n_dp):
                qo, so = oracle.quantize_int8(out_ref[o * S:(o + 1) * S], 256)
                assert np.array_equal(q.q[o].cpu().numpy(), qo)
                assert np.array_equal(q.scales[o, :q.nb].cpu().numpy(), so)
        else:
            assert np.array_equal(parity.bits(u.shards).reshape(-1), out_ref)
    assert eng.ring.resident == 0 and eng.ring.peak <= 2


def test_engines_follow_the_scheduler(zlib, cuda_device):
    """WarmupDecayLR ("DeepSpeed ZeRO", "The configuration file"): every step's
    lr from the schedule, the update bit-exact against the oracle at that lr."""
    from oracle import formulas
    sched = {"type": "WarmupDecayLR", "params": {"warmup_min_lr": 1e-5, "warmup_max_lr": 1e-3,
                                                 "warmup_num_steps": 2, "total_num_steps": 4}}
    n_dp, N = 4, 50_001
    cfg = ZeroConfig.from_dict({"zero_optimization": {"stage": 2},
                                "optimizer": {"type": "AdamW", "params": {
                                    "lr": HP.lr, "betas": [HP.beta1, HP.beta2], "eps": HP.eps,
                                    "weight_decay": HP.weight_decay}},
                                "scheduler": sched})
    eng = ZeroEngine([N], n_dp, cfg, master=inputs.master_weights(N, 50_016, seed=5).cuda())
    P = eng.L.padded_n
    units = [[7_001], [30_000, 13]]
    eng3 = Zero3Engine(units, n_dp, ZeroConfig.from_dict({**{"zero_optimization": {"stage": 3}},
                                                         "optimizer": cfg_opt(), "scheduler": sched}))
    state = [parity.f32(eng.master), np.zeros(P, np.float32), np.zeros(P, np.float32)]
    states3 = [[parity.f32(u.master), np.zeros(u.layout.padded_n, np.float32),
                np.zeros(u.layout.padded_n, np.float32)] for u in eng3.units]
    for t in range(1, 6):                      # past total_num_steps: lr 0, decay still 0
        hp = oracle.AdamW(lr=formulas.warmup_decay_lr(t, 1e-5, 1e-3, 2, 4), beta1=HP.beta1, beta2=HP.beta2,
                          eps=HP.eps, weight_decay=HP.weight_decay)
        g = inputs.grads_bf16(n_dp, N, P, seed=6, step=t)
        eng.backward(g.cuda())
        eng.step()
        for i, u in enumerate(eng3.units):
            g3 = inputs.grads_bf16(n_dp, u.layout.n, u.layout.padded_n, seed=7 + i, step=t)
            eng3.backward(i, g3.cuda())
            out3, *states3[i] = oracle.rs_adamw_reference(parity.bits(g3), n_dp, *states3[i], hp, t)
            torch.cuda.synchronize()
            parity.assert_state([u.master, u.m, u.v], states3[i], what=f"unit {i} t={t} ")
            assert np.array_equal(parity.bits(u.shards).reshape(-1), out3)
        eng3.step()
        torch.cuda.synchronize()
        out_ref, *state = oracle.rs_adamw_reference(parity.bits(g), n_dp, *state, hp, t)
        parity.assert_state([eng.master, eng.m, eng.v], state, what=f"t={t} ")
        assert np.array_equal(parity.bits(eng.weights), out_ref)


def cfg_opt():
    return {"type": "AdamW", "params": {"lr": HP.lr, "betas": [HP.beta1, HP.beta2], "eps": HP.eps,
                                        "weight_decay": HP.weight_decay}}


@pytest.mark.parametrize("qw", [False, True])
def test_zero3_engine_overlap_comm(zlib, cuda_device, qw):
    """overlap_comm: every gather after the first is served from a prefetch one
    unit ahead on a side stream; the gathered weights and the step's state are
    bit-identical to the engine without it, with at most two units resident."""
    n_dp = 4
    units = [[4097], [33_031], [1000, 24, 3, 5000], [77]]

    def run(overlap):
        cfg = ZeroConfig.from_dict({"zero_optimization": {"stage": 3, "overlap_comm": overlap,
                                                          "zero_quantized_weights": qw},
                                    "optimizer": cfg_opt()})
        eng = Zero3Engine(units, n_dp, cfg)
        for i, u in enumerate(eng.units):
            u.master.copy_(inputs.master_weights(u.layout.n, u.layout.padded_n, seed=40 + i).cuda())
            zlib.zero_cast_bf16(u.master, u.shards.view(-1))
            if eng.q8 is not None:
                zstep.zero3_quantize(u, eng.q8[i])
        seen, served = [], 0
        for t in (1, 2):
            for i in range(len(units)):
                served += int(eng.pf is not None and ("fwd", i) in eng.pf.pending)
                seen.append(eng.gather(i, "fwd").clone())
                eng.release(i, "fwd")
            for i in reversed(range(len(units))):
                served += int(eng.pf is not None and ("bwd", i) in eng.pf.pending)
                seen.append(eng.gather(i, "bwd").clone())
                eng.release(i, "bwd")
                u = eng.units[i]
                eng.backward(i, inputs.grads_bf16(n_dp, u.layout.n, u.layout.padded_n, seed=50 + i,
                                                  step=t).cuda())
            eng.step()
        torch.cuda.synchronize()
        assert eng.ring.peak <= 2 and eng.ring.resident == 0
        return eng, seen, served

    a, seen_a, served_a = run(False)
    b, seen_b, served_b = run(True)
    assert served_a == 0 and served_b == 2 * (2 * len(units) - 1)     # all but each step's first gather
    assert not b.pf.pending
    for x, y in zip(seen_a, seen_b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for ua, ub in zip(a.units, b.units):
        for x, y in ((ua.master, ub.master), (ua.m, ub.m), (ua.v, ub.v), (ua.shards, ub.shards)):
            assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16),
                               y.view(torch.int32) if y.dtype == torch.float32 else y.view(torch.int16))
    # both against the oracle's stage-3 sequence from the same initial state
    layouts = [u.layout for u in b.units]
    init_w = [inputs.master_weights(L.n, L.padded_n, seed=40 + i).numpy() for i, L in enumerate(layouts)]
    gathered, st, sh = parity.zero3_oracle_run(
        [[w, np.zeros_like(w), np.zeros_like(w)] for w in init_w], [oracle.cast_bf16(w) for w in init_w],
        [lambda t, i=i, L=L: parity.bits(inputs.grads_bf16(n_dp, L.n, L.padded_n, seed=50 + i, step=t))
         for i, L in enumerate(layouts)], HP, (1, 2), n_dp, 256 if qw else None)
    assert len(gathered) == len(seen_b)
    for x, (p, i, ref) in zip(seen_b, gathered):
        assert np.array_equal(parity.bits(x), ref), (p, i)
    if qw:          # the 8-bit update writes only the 8-bit shards: bring the bf16 ones up to date
        b._bf16_shards_current()
    for i, ub in enumerate(b.units):
        parity.assert_state([ub.master, ub.m, ub.v], st[i], what=f"unit {i} ")
        assert np.array_equal(parity.bits(ub.shards).reshape(-1), sh[i])


def _cfg_dict(stage, **zo):
    return {"zero_optimization": {"stage": stage, **zo}, "optimizer": cfg_opt()}


def test_zero12_engine_checkpoint_resume_and_16bit_model(zlib, cuda_device, tmp_path):
    """Two steps, save, a fresh engine loads and both take a third step: the
    same state bit for bit.  The 16-bit model file holds the engine's bf16
    weights without padding, split at the tensors' boundaries."""
    from zero_sharded_mixed_gb300 import checkpoint as ck
    n_dp, numels = 4, [30_001, 7, 20_000]
    cfg = ZeroConfig.from_dict(_cfg_dict(2))
    N = sum(numels)
    a = ZeroEngine(numels, n_dp, cfg, master=inputs.master_weights(N, 50_016, seed=3).cuda())
    P = a.L.padded_n
    grads = lambda t: inputs.grads_bf16(n_dp, N, P, seed=8, step=t).cuda()
    for t in (1, 2):
        a.backward(grads(t))
        a.step()
    a.save_checkpoint(str(tmp_path / "ck"))
    a.save_16bit_model(str(tmp_path / "w16"))
    b = ZeroEngine(numels, n_dp, cfg)
    assert b.load_checkpoint(str(tmp_path / "ck")) == 2
    for e in (a, b):
        e.backward(grads(3))
        e.step()
    torch.cuda.synchronize()
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(a.weights.view(torch.int16), b.weights.view(torch.int16))
    w16 = ck.load_16bit_model(str(tmp_path / "w16"), split=True)
    assert [len(x) for x in w16] == numels
    # the file holds the weights after step 2: recompute them from the oracle's step
    state = [parity.f32(inputs.master_weights(N, 50_016, seed=3)), np.zeros(P, np.float32),
             np.zeros(P, np.float32)]
    for t in (1, 2):
        out_ref, *state = oracle.rs_adamw_reference(parity.bits(grads(t)), n_dp, *state, HP, t)
    assert np.array_equal(np.concatenate(w16), out_ref[:N])


@pytest.mark.parametrize("qw", [False, True])
def test_zero3_engine_checkpoint_resume_and_16bit_model(zlib, cuda_device, tmp_path, qw):
    from zero_sharded_mixed_gb300 import checkpoint as ck
    n_dp = 4
    units = [[4097], [33_031], [1000, 24, 3, 5000]]
    zo = {"zero_quantized_weights": qw, "stage3_gather_16bit_weights_on_model_save": True}
    cfg = ZeroConfig.from_dict(_cfg_dict(3, **zo))

    def engine():
        e = Zero3Engine(units, n_dp, cfg)
        for i, u in enumerate(e.units):
            u.master.copy_(inputs.master_weights(u.layout.n, u.layout.padded_n, seed=60 + i).cuda())
            u.shards.view(-1).copy_(u.master.to(torch.bfloat16))
            if e.q8 is not None:
                zstep.zero3_quantize(u, e.q8[i])
        return e

    def step(e, t):
        for i in reversed(range(len(units))):
            u = e.units[i]
            e.gather(i, "bwd")
            e.release(i, "bwd")
            e.backward(i, inputs.grads_bf16(n_dp, u.layout.n, u.layout.padded_n, seed=70 + i, step=t).cuda())
        e.step()

    a = engine()
    step(a, 1)
    a.save_checkpoint(str(tmp_path / "ck"))
    a.save_16bit_model(str(tmp_path / "w16"))
    b = Zero3Engine(units, n_dp, cfg)
    assert b.load_checkpoint(str(tmp_path / "ck")) == 1
    step(a, 2)
    step(b, 2)
    torch.cuda.synchronize()
    for ua, ub in zip(a.units, b.units):
        for x, y in ((ua.master, ub.master), (ua.m, ub.m), (ua.v, ub.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    if qw:
        for qa, qb in zip(a.q8, b.q8):
            assert torch.equal(qa.q, qb.q) and torch.equal(qa.scales, qb.scales)
    w16 = ck.load_16bit_model(str(tmp_path / "w16"))
    masters = np.concatenate([ck.consolidate(str(tmp_path / "ck" / f"unit_{i:05d}"))["master"]
                              for i in range(len(units))])
    assert np.array_equal(w16, oracle.cast_bf16(masters))
    plain = Zero3Engine(units, n_dp, ZeroConfig.from_dict(_cfg_dict(3)))
    with pytest.raises(RuntimeError):
        plain.save_16bit_model(str(tmp_path / "refused"))


def test_engine_tracing(zlib, cuda_device):
    """Step time, the gradient norm (with clipping) against the oracle, and the
    memory estimate by the pages' formula."""
    n_dp, N = 4, 100_003
    cfg = ZeroConfig.from_dict({**_cfg_dict(2), "gradient_clipping": 1.0})
    eng = ZeroEngine([N], n_dp, cfg, master=inputs.master_weights(N, 100_032, seed=1).cuda())
    assert eng.last_step_ms() is None and eng.grad_norm() is None
    P = eng.L.padded_n
    g = inputs.grads_bf16(n_dp, N, P, seed=2, step=1, std=1.0)
    eng.backward(g.cuda())
    eng.step()
    assert eng.last_step_ms() > 0
    ref = oracle.grad_norm_sq(parity.bits(g), n_dp) ** 0.5
    assert abs(eng.grad_norm() - ref) <= 1e-9 * ref
    est = eng.memory_estimate()
    assert est["params"] == N
    assert est["stage0"] == 16 * N and abs(est["stage2"] - (2 * N + 14 * N / n_dp)) < 1e-6 * N
    assert abs(est["stage3"] - 16 * N / n_dp) < 1e-6 * N
    assert est["this_process_bytes"] >= P * 12 + P * 2
    z3 = Zero3Engine([[4097], [33_031]], n_dp, ZeroConfig.from_dict(_cfg_dict(3)))
    assert z3.memory_estimate()["params"] == 4097 + 33_031 and z3.grad_norm() is None
