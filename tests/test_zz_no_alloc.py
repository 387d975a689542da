"""The norm entry point that allocates nothing (zero_grad_norm_sq_static),
checked against the workspace version (zero_grad_norm_sq) through the C ABI.

It exists for callers that cannot allocate device memory themselves -- a
plugin handed only its inputs and outputs by a framework that owns every
device allocation, or a path where cudaMalloc's implicit synchronization is
not allowed.  Its partial sums live in a fixed array inside the library, shared
by every call; two calls in a row check that nothing left over from the first
call reaches the second.  This file is collected last, so a run that stops at
the first failure has run every other test before it."""
import numpy as np
import pytest
import torch

import oracle
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu


def _sources(zb, n_src, N, dtype, seed):
    rng = np.random.default_rng(seed)
    xf = (rng.standard_normal((n_src, N)) * 1e-2).astype(np.float32)
    if dtype == "bf16":
        xb = oracle.cast_bf16(xf)
        return [inputs.from_bf16_bits(xb[r], "cuda") for r in range(n_src)], zb.ZERO_BF16
    return [torch.from_numpy(xf[r].copy()).cuda() for r in range(n_src)], zb.ZERO_F32


def test_static_scratch_matches_workspace_version(zlib, cuda_device):
    zb = zlib
    bufs = zstep.NormBuffers("cuda")
    got = torch.zeros(1, dtype=torch.float64, device="cuda")
    # two calls in a row, different sizes and source kinds: the second must not
    # see anything the first left in the shared array
    cases = [(8, 3_000_017, "bf16", 1), (2, 40_001, "f32", 2)]
    for n_src, N, dtype, seed in cases:
        L = zb.zero_layout([N], 1, align=1)
        srcs, code = _sources(zb, n_src, N, dtype, seed)
        zb.zero_grad_norm_sq(L, srcs, code, 0, float(n_src), 0, N, bufs.workspace, bufs.norm_sq, False)
        zb.zero_grad_norm_sq_static(L, srcs, code, 0, float(n_src), 0, N, got, False)
        torch.cuda.synchronize()
        ref, val = float(bufs.norm_sq.item()), float(got.item())
        assert val == pytest.approx(ref, rel=1e-12)
        assert val == ref        # same kernels, same grid: the same bits
    # accumulating over two pieces agrees as well
    n_src, N = 4, 1_000_003
    L = zb.zero_layout([N], 1, align=1)
    srcs, code = _sources(zb, n_src, N, "bf16", 3)
    for j, (s, e) in enumerate([(0, 400_000), (400_000, N)]):
        zb.zero_grad_norm_sq(L, srcs, code, 0, float(n_src), s, e, bufs.workspace, bufs.norm_sq, j > 0)
        zb.zero_grad_norm_sq_static(L, srcs, code, 0, float(n_src), s, e, got, j > 0)
    torch.cuda.synchronize()
    assert float(got.item()) == pytest.approx(float(bufs.norm_sq.item()), rel=1e-12)
