"""Parity of the 8-bit quantized weight gather (zero_quantize_int8,
zero_gather_layer_int8) with the oracle, bit for bit, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu


def _oracle_unit(shards_bits, block):
    """Per-rank oracle quantization, then the dequantized concatenation."""
    qs, ss, full = [], [], []
    for row in shards_bits:
        q, s = oracle.quantize_int8(row, block)
        qs.append(q)
        ss.append(s)
        full.append(oracle.dequantize_int8(q, s, block))
    return qs, ss, np.concatenate(full)


@pytest.mark.parametrize("numels,n_dp,align,block", [
    ([4096], 1, 8, 256), ([100_003], 3, 8, 256), ([33_031, 7, 1], 7, 8, 512),
    ([1_000_000], 8, 8, 1024), ([5_000_011], 8, 8, 2048), ([4097], 5, 1, 256), ([77], 3, 1, 256),
])
def test_quantize_and_gather_bit_exact(zlib, cuda_device, numels, n_dp, align, block):
    zb = zlib
    L = zb.zero_layout(numels, n_dp, align=align)
    w = inputs.master_weights(L.n, L.padded_n, seed=n_dp)
    shards = w.to(torch.bfloat16).cuda()
    unit = zstep.Zero3Unit(L, shards.view(n_dp, L.shard), None, None, None)
    qs = zstep.Int8Shards(L, block)
    zstep.zero3_quantize(unit, qs)
    ring = zstep.GatherRing(L.padded_n)
    buf = zstep.zero3_gather_int8(unit, qs, ring, "u")
    torch.cuda.synchronize()
    ref_q, ref_s, ref_full = _oracle_unit(parity.bits(shards).reshape(n_dp, L.shard), block)
    np.testing.assert_array_equal(qs.q.cpu().numpy(), np.stack(ref_q))
    np.testing.assert_array_equal(qs.scales[:, :qs.nb].cpu().numpy(), np.stack(ref_s))
    assert np.array_equal(parity.bits(buf), ref_full)
    # the gathered unit is within half a quantization step (+ a bf16 half-ulp) of the bf16 unit
    x = oracle.bf16_to_f32(parity.bits(shards)).astype(np.float64)
    y = oracle.bf16_to_f32(ref_full).astype(np.float64)
    step = np.concatenate([np.repeat(s.astype(np.float64), block)[:L.shard] for s in ref_s])
    assert np.all(np.abs(y - x) <= step / 2 * (1 + 1e-6) + np.abs(y) * 2.0 ** -8 + 1e-45)
    ring.release("u")


def test_special_blocks(zlib, cuda_device):
    """An all-zero block, exact ties, the block maximum at +-127, mixed signs."""
    zb = zlib
    vals = np.zeros(1024, np.float32)
    vals[:6] = [127.0, 0.5, 1.5, 2.5, -2.5, 3.5]              # scale 1: ties to even
    vals[256:512] = np.linspace(-3.0, 3.0, 256, dtype=np.float32)
    vals[768:1024] = -np.float32(1e-3) * np.arange(256, dtype=np.float32)
    bits = oracle.cast_bf16(vals)
    L = zb.zero_layout([1024], 1)
    shards = inputs.from_bf16_bits(bits, "cuda")
    unit = zstep.Zero3Unit(L, shards.view(1, 1024), None, None, None)
    qs = zstep.Int8Shards(L, 256)
    zstep.zero3_quantize(unit, qs)
    full = torch.empty(1024, dtype=torch.bfloat16, device="cuda")
    zb.zero_gather_layer_int8(L, [qs.q[0]], [qs.scales[0]], full, 256)
    torch.cuda.synchronize()
    rq, rs = oracle.quantize_int8(bits, 256)
    np.testing.assert_array_equal(qs.q[0].cpu().numpy(), rq)
    np.testing.assert_array_equal(qs.scales[0].cpu().numpy(), rs)
    assert np.array_equal(parity.bits(full), oracle.dequantize_int8(rq, rs, 256))
    assert list(rq[:6]) == [127, 0, 2, 2, -2, 4] and rs[2] == 0.0


def test_quantized_zero3_step_sequence(zlib, cuda_device):
    """Stage 3 with 8-bit gathers over ragged units at n_dp = 8: quantize the
    shards, gather twice (forward, backward), reduce-scatter, update the bf16
    shards, re-quantize; each gathered unit equals the oracle's dequantized
    concatenation of the current shards."""
    zb = zlib
    n_dp = 8
    hp = oracle.AdamW()
    for i, numels in enumerate([[4097], [1000, 24, 3, 5000], [262_144]]):
        L = zb.zero_layout(numels, n_dp)
        P = L.padded_n
        w = inputs.master_weights(L.n, P, seed=40 + i).cuda()
        shards = w.to(torch.bfloat16)
        unit = zstep.Zero3Unit(L, shards.view(n_dp, L.shard), w, torch.zeros(P, device="cuda"),
                               torch.zeros(P, device="cuda"))
        qs = zstep.Int8Shards(L, 256)
        ring = zstep.GatherRing(P)
        A = torch.empty(P, device="cuda")
        for t in (1, 2):
            zstep.zero3_quantize(unit, qs)
            ref = _oracle_unit(parity.bits(unit.shards), 256)[2]
            for phase in ("fwd", "bwd"):
                buf = zstep.zero3_gather_int8(unit, qs, ring, phase)
                torch.cuda.synchronize()
                assert np.array_equal(parity.bits(buf), ref)
                ring.release(phase)
            g = inputs.grads_bf16(n_dp, L.n, P, seed=50 + i, step=t)
            zstep.zero3_layer_reduce_scatter(unit, [g[r].cuda() for r in range(n_dp)], A)
            zstep.zero3_update(unit, A, zb.ZeroAdamW.make(hp.lr, hp.beta1, hp.beta2, hp.eps,
                                                          hp.weight_decay, t))
        torch.cuda.synchronize()
        assert ring.peak <= 1
        # a receiver gets 1 byte per weight plus 4 bytes per block, instead of 2 per weight
        assert qs.wire_bytes() == P + n_dp * qs.nb * 4
        if L.shard % 256 == 0:
            assert qs.wire_bytes() == pytest.approx(P * (1 + 4 / 256))
