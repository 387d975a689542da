"""The norm entry point that allocates nothing (zero_grad_norm_sq_static),
checked through the C ABI against the workspace version (zero_grad_norm_sq)
and against the oracle's fp64 norm of the mean gradient.

It exists for callers that cannot allocate device memory themselves -- a
plugin handed only its inputs and outputs by a framework that owns every
device allocation, or a path where cudaMalloc's implicit synchronization is
not allowed.  Its partial sums live in a fixed array inside the library, shared
by every call; calls in a row check that nothing left over from one call
reaches the next.  The array is sized from the partial pass's bound on
resident CTAs, so a build with smaller CTAs (more partials per SM) works too:
a 128-thread build is checked in a child process of its own.  This file is
collected last, so a run that stops at the first failure has run every other
test before it."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (n_src = n_dp, N, dtype, seed): ragged lengths, rank counts 1, 3 and 8, both
# source kinds; run in this order, back to back, on the one shared array
CASES = [(8, 3_000_017, "bf16", 1), (3, 40_001, "f32", 2), (1, 1_048_583, "bf16", 3),
         (8, 77_777, "f32", 4), (3, 2_000_003, "bf16", 5)]


def _sources(zb, n_src, N, dtype, seed):
    import torch

    import oracle
    from zero_sharded_mixed_gb300 import inputs
    rng = np.random.default_rng(seed)
    xf = (rng.standard_normal((n_src, N)) * 1e-2).astype(np.float32)
    if dtype == "bf16":
        xb = oracle.cast_bf16(xf)
        return [inputs.from_bf16_bits(xb[r], "cuda") for r in range(n_src)], zb.ZERO_BF16, xb
    return [torch.from_numpy(xf[r].copy()).cuda() for r in range(n_src)], zb.ZERO_F32, xf


def check_static_norm(zb):
    """Every case: the static entry point's norm equals the workspace entry
    point's bit for bit (same kernels, same grid) and the oracle's within
    1e-12 relative; then a norm accumulated over two pieces of one range."""
    import torch

    import oracle
    from zero_sharded_mixed_gb300 import step as zstep
    bufs = zstep.NormBuffers("cuda")
    got = torch.zeros(1, dtype=torch.float64, device="cuda")
    for n_src, N, dtype, seed in CASES:
        L = zb.zero_layout([N], 1, align=1)
        srcs, code, host = _sources(zb, n_src, N, dtype, seed)
        zb.zero_grad_norm_sq(L, srcs, code, 0, float(n_src), 0, N, bufs.workspace, bufs.norm_sq, False)
        zb.zero_grad_norm_sq_static(L, srcs, code, 0, float(n_src), 0, N, got, False)
        torch.cuda.synchronize()
        ref, val = float(bufs.norm_sq.item()), float(got.item())
        exact = oracle.grad_norm_sq(host, n_src)
        assert val == ref, (n_src, N, dtype)
        assert val == pytest.approx(exact, rel=1e-12), (n_src, N, dtype)
    # accumulating over two pieces of one range agrees as well
    n_src, N = 4, 1_000_003
    L = zb.zero_layout([N], 1, align=1)
    srcs, code, host = _sources(zb, n_src, N, "bf16", 6)
    for j, (s, e) in enumerate([(0, 400_000), (400_000, N)]):
        zb.zero_grad_norm_sq(L, srcs, code, 0, float(n_src), s, e, bufs.workspace, bufs.norm_sq, j > 0)
        zb.zero_grad_norm_sq_static(L, srcs, code, 0, float(n_src), s, e, got, j > 0)
    torch.cuda.synchronize()
    assert float(got.item()) == pytest.approx(float(bufs.norm_sq.item()), rel=1e-12)
    assert float(got.item()) == pytest.approx(oracle.grad_norm_sq(host, n_src), rel=1e-12)


def test_static_scratch_matches_workspace_version_and_oracle(zlib, cuda_device):
    check_static_norm(zlib)


def test_static_scratch_in_a_128_thread_build(tmp_path, cuda_device):
    """A build with 128-thread CTAs launches up to 16 partial-pass CTAs per SM,
    so its static array holds 512 x 16 partials; the entry point must accept
    this GPU and give the same results."""
    from zero_sharded_mixed_gb300 import build as zbuild
    lib = zbuild.build(defines=["ZGB_THREADS=128"], out=str(tmp_path / "libzero_gb300_t128.so"))
    r = subprocess.run([sys.executable, os.path.abspath(__file__), lib], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ALL OK" in r.stdout, r.stdout


def _child(lib: str) -> None:
    sys.path.insert(0, ROOT)
    from zero_sharded_mixed_gb300 import binding as zb
    zb.lib_path = lib
    zb._lib = None
    zb.load()
    check_static_norm(zb)
    print("ALL OK")


if __name__ == "__main__":
    _child(sys.argv[1])
