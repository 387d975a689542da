"""Checkpoint and resume on the GPU: a run saved after two steps, restored into
fresh device buffers and continued, ends bit-identical to the same run without
the interruption; a resharded checkpoint resumes at another rank count."""
import numpy as np
import pytest
import torch

from tests import parity
from zero_sharded_mixed_gb300 import checkpoint as ck
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu


def _run(zb, L, state, out, t0, t1):
    for t in range(t0, t1):
        g = inputs.grads_bf16(L.n_dp, L.n, L.padded_n, seed=8, step=t)
        zstep.zero12_step(L, [g[r].cuda() for r in range(L.n_dp)], *state, out,
                          zb.ZeroAdamW.make(step=t))


def test_save_restore_continue(zlib, cuda_device, tmp_path):
    zb = zlib
    numels = [300_000, 17, 99_999]
    L = zb.zero_layout(numels, 4, bucket_elems=100_000)
    P = L.padded_n
    w0 = inputs.master_weights(L.n, P, seed=8).cuda()
    ref = [w0.clone(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    ref_out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    _run(zb, L, ref, ref_out, 1, 5)
    st = [w0.clone(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    _run(zb, L, st, out, 1, 3)
    ck.save(str(tmp_path / "c"), L, numels, *st, 2, zb.ZeroAdamW.make(step=2), out_bf16=out)
    fresh = [torch.full((P,), float("nan"), device="cuda") for _ in range(3)]
    fresh_out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    t = ck.restore(str(tmp_path / "c"), L, *fresh, out_bf16=fresh_out)
    assert t == 2
    assert torch.equal(fresh_out.view(torch.int16), out.view(torch.int16))
    _run(zb, L, fresh, fresh_out, t + 1, 5)
    torch.cuda.synchronize()
    for a, b in zip(fresh, ref):
        parity.assert_bit_exact_f32(a, b)
    assert torch.equal(fresh_out.view(torch.int16), ref_out.view(torch.int16))
    # resharded to 3 ranks, the state restores into the 3-rank layout element for element
    ck.reshard(str(tmp_path / "c"), str(tmp_path / "d"), 3)
    L3 = zb.zero_layout(numels, 3, bucket_elems=100_000)
    st3 = [torch.zeros(L3.padded_n, device="cuda") for _ in range(3)]
    assert ck.restore(str(tmp_path / "d"), L3, *st3) == 2
    for a3, a in zip(st3, st):
        np.testing.assert_array_equal(parity.f32(a3)[:L.n], parity.f32(a)[:L.n])
    # and a step at 3 ranks runs on it
    out3 = torch.zeros(L3.padded_n, dtype=torch.bfloat16, device="cuda")
    _run(zb, L3, st3, out3, 3, 4)
    torch.cuda.synchronize()
    assert torch.isfinite(st3[0]).all()
