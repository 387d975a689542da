"""Comparison helpers for the CUDA-vs-oracle parity tests.

Tolerances are the contract for this path: fp32 master / m / v within
1e-6 relative + 1e-9 absolute of the oracle, bf16 weights within 1 bf16 ulp,
layouts and offsets bit-exact.  Because both sides use the same operation
order with IEEE rounding and no FMA contraction, the tests also record how many
elements match bit for bit (expected: all of them).
"""
from __future__ import annotations

import numpy as np
import torch

RTOL = 1e-6
ATOL = 1e-9
BF16_ULPS = 1


def f32(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").contiguous().numpy().astype(np.float32, copy=False)
    return np.asarray(t, np.float32)


def bits(t) -> np.ndarray:
    """bf16 tensor (or uint16 array) -> uint16 bit patterns on the host."""
    if isinstance(t, torch.Tensor):
        assert t.dtype == torch.bfloat16
        return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.asarray(t, np.uint16)


def _nan_bf16(h):
    return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)


def _ordered(h):
    h = h.astype(np.int32)
    return np.where(h & 0x8000, -(h & 0x7FFF), h)


def assert_bf16_close(got, ref, ulps=BF16_ULPS, what="bf16"):
    g, r = bits(got), bits(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    gn, rn = _nan_bf16(g), _nan_bf16(r)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    d = np.abs(_ordered(g[~gn]) - _ordered(r[~rn]))
    worst = int(d.max()) if d.size else 0
    assert worst <= ulps, f"{what}: {int((d > ulps).sum())} elements beyond {ulps} ulp (worst {worst})"
    return int((g == r).sum())


def assert_f32_close(got, ref, rtol=RTOL, atol=ATOL, what="fp32"):
    g, r = f32(got), f32(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    gn, rn = np.isnan(g), np.isnan(r)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    with np.errstate(invalid="ignore"):    # inf - inf: equal infinities are accepted below
        ok = np.abs(g[~gn].astype(np.float64) - r[~rn]) <= atol + rtol * np.abs(r[~rn].astype(np.float64))
    ok |= (g[~gn] == r[~rn])   # equal infinities
    assert ok.all(), (f"{what}: {int((~ok).sum())} of {ok.size} elements outside "
                      f"{rtol} rel + {atol} abs")
    return int((g.view(np.uint32) == r.view(np.uint32)).sum())


def assert_bit_exact_f32(got, ref, what="fp32"):
    g, r = f32(got), f32(ref)
    same = (g.view(np.uint32) == r.view(np.uint32)) | (np.isnan(g) & np.isnan(r))
    assert same.all(), f"{what}: {int((~same).sum())} of {same.size} elements differ in some bit"


def assert_state(got_wmv, ref_wmv, exact=True, what=""):
    for name, g, r in zip("wmv", got_wmv, ref_wmv):
        assert_f32_close(g, r, what=f"{what}{name}")
        if exact:
            assert_bit_exact_f32(g, r, what=f"{what}{name}")


def zero3_oracle_run(states, shards, grads, hp, steps, n_dp, block=None):
    """The oracle's statement of the stage-3 step sequence over a list of
    units, on the host: per step t, every unit gathered for forward in order,
    then in reverse every unit gathered for backward, its gradient
    reduce-scattered (fp32 sum over ranks) and its owned shards updated, bf16
    into the owners' shards ("ZeRO and FSDP", "FSDP, ZeRO-3 inside PyTorch";
    "DeepSpeed ZeRO", "Stage 3 step by step").  With block set, the weights
    travel as 8-bit shards: each owner's bf16 shard is quantized after every
    update and the gathers dequantize ("ZeRO and FSDP", "Fewer bytes on the
    wire").

    states[i] = [w, m, v] fp32 arrays (padded length), shards[i] the bf16 bit
    patterns (padded length), grads[i](t) the (n_dp, P) bf16 bit patterns of
    unit i's gradient at step t.  Returns (gathered, states, shards):
    gathered = [(phase, i, bits)] in gather order; states and shards are new
    arrays (the inputs are not modified)."""
    import oracle
    states = [[np.asarray(x, np.float32).copy() for x in st] for st in states]
    shards = [np.asarray(s, np.uint16).copy() for s in shards]

    def quant(s):
        return [oracle.quantize_int8(o, block) for o in s.reshape(n_dp, -1)]

    q = [quant(s) for s in shards] if block else None

    def gather(i):
        if block:
            return oracle.all_gather(np.stack([oracle.dequantize_int8(qq, sc, block) for qq, sc in q[i]]))
        return oracle.all_gather(shards[i].reshape(n_dp, -1))

    gathered = []
    for t in steps:
        for i in range(len(states)):
            gathered.append(("fwd", i, gather(i)))
        for i in reversed(range(len(states))):
            gathered.append(("bwd", i, gather(i)))
            A = oracle.accumulate_reduce(None, grads[i](t), first=True)
            out, *states[i] = oracle.rs_adamw_reference(A[None, :], n_dp, *states[i], hp, t)
            shards[i] = out
            if block:
                q[i] = quant(out)
    return gathered, states, shards
