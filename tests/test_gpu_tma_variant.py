"""Parity of the TMA-staged build of the fused update against the oracle.

The library built with ZGB_RS_TMA=1 sends bf16-source updates with 1, 2, 4 or
8 sources through the bulk-copy kernels instead of the register-staged one:
the warp-specialized pipeline (rs_adamw_ws_kernel, the default) and, with
ZGB_TMA_WS=0, the CTA-synchronous ring (rs_adamw_tma_kernel).  It is an opt-in build, so this test compiles it into a temporary
library and checks it in a child process of its own (one library per
process), bit for bit against the oracle: several steps, several buckets,
ranges that span many 1024-element tiles with a ragged last tile, a range
whose length is not a multiple of 8, a range shorter than 8 elements, a source count the TMA kernel does not take (3: the
register-staged fallback inside the same build), and the clipped update."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("defines", [["ZGB_RS_TMA=1"], ["ZGB_RS_TMA=1", "ZGB_TMA_WS=0"]],
                         ids=["warp-specialized", "cta-synchronous"])
def test_tma_build_matches_the_oracle(tmp_path, cuda_device, defines):
    from zero_sharded_mixed_gb300 import build as zbuild
    lib = zbuild.build(defines=defines, out=str(tmp_path / "libzero_gb300_tma.so"))
    r = subprocess.run([sys.executable, os.path.abspath(__file__), lib], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ALL OK" in r.stdout, r.stdout


def _child(lib: str) -> None:
    import numpy as np
    import torch

    sys.path.insert(0, ROOT)
    import oracle
    from tests import parity
    from zero_sharded_mixed_gb300 import binding as zb
    from zero_sharded_mixed_gb300 import inputs
    from zero_sharded_mixed_gb300 import step as zstep

    zb.lib_path = lib
    zb._lib = None
    zb.load()
    hp_o = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)

    def hp(t):
        return zb.ZeroAdamW.make(hp_o.lr, hp_o.beta1, hp_o.beta2, hp_o.eps, hp_o.weight_decay, t)

    def case(N, n_dp, bucket, steps, clip=None, seed=0):
        L = zb.zero_layout([N], n_dp, bucket_elems=bucket)
        P = L.padded_n
        w0 = inputs.master_weights(N, P, seed=seed)
        st = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
        out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
        ref = [parity.f32(w0), np.zeros(P, np.float32), np.zeros(P, np.float32)]
        bufs = zstep.NormBuffers("cuda") if clip else None
        for t in range(1, steps + 1):
            g = inputs.grads_bf16(n_dp, N, P, seed=seed, step=t, std=1.0 if clip else 1e-3)
            gd = [g[r].cuda() for r in range(n_dp)]
            gb = parity.bits(g)
            if clip:
                zstep.zero12_step_clipped(L, gd, *st, out, hp(t), clip, bufs)
                nsq = oracle.grad_norm_sq(gb, n_dp)
                ref_out, *ref = oracle.rs_adamw_reference(gb, n_dp, *ref, hp_o, t, clip=(nsq, clip))
            else:
                zstep.zero12_step(L, gd, *st, out, hp(t))
                ref_out, *ref = oracle.rs_adamw_reference(gb, n_dp, *ref, hp_o, t)
            torch.cuda.synchronize()
            what = f"N={N} n_dp={n_dp} bucket={bucket} t={t} clip={clip}: "
            parity.assert_state(st, ref, what=what)
            assert np.array_equal(parity.bits(out), ref_out), what + "bf16 output"
        print("ok", N, n_dp, bucket, clip, flush=True)

    for n_dp in (1, 2, 4, 8):
        case(37 * 1024 * n_dp - 5, n_dp, 30_000, 3)          # many tiles, ragged tail, buckets
    case(200_003, 8, 500_000_000, 2)                         # one bucket, tail of 3 in the last shard
    case(5, 1, 500_000_000, 2)                               # shorter than one 8-element vector
    case(100_003, 3, 30_000, 2)                              # 3 sources: register-staged fallback
    case(100_003, 4, 30_004, 2)                              # first bucket ends in a 4-element tail;
                                                             # later ones are not 16-byte aligned
    case(100_003, 4, 30_000, 2, clip=1.0)                    # clipped update through the TMA kernel
    zb.zero_status_check(None)                            # raises on a CUDA error or a timeout
    print("ALL OK", flush=True)


if __name__ == "__main__":
    _child(sys.argv[1])
