"""Edge cases of the 8-bit gradient kernels against the oracle, bit for bit,
through the C ABI, in the default build and in the opt-in build with
bulk-copy staging of the code streams (ZGB_QWS=3).

The opt-in build sends an 8-bit gradient launch with 1, 2, 4 or 8 sources to
the warp-specialized kernel when every source's slice starts on a 16-byte
boundary, and to the register-staged kernel otherwise.  The cases are chosen
for the staged kernel's edges: slices of several 2048-element tiles per CTA
with a partial last tile and a tail of fewer than 16 elements; layouts whose
odd owners' slices start 8 bytes off the 16-byte grid, so that one call mixes
both kernels; calls over whole shards (one launch, blockIdx.y = owner) and over
ranges that cut shards; the overwrite and the add of the accumulation; every
staged source count; the update with bf16 and with 8-bit output.  The opt-in
build runs this file's cases in a child process of its own (one library per
process)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

HP = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
BLOCK = 256


def _hp(zb, t):
    return zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, t)


def _quantize(zb, L, g, block=BLOCK):
    qg = zstep.Int8Grads(L, g.shape[0], block)
    qg.quantize([g[r].cuda() for r in range(g.shape[0])])
    q_ref, s_ref = oracle.quantize_grad_int8(parity.bits(g), L.n_dp, block)
    return qg, q_ref, s_ref


# (N, n_dp, align): S = 81,920 (40 tiles, 16-byte aligned slices); S = 1,000,008
# (odd owners 8 bytes off the grid); S = 66,664 with a ragged N (partial tiles,
# tails); one tile and a bit; fewer elements than one vector per owner
CASES = [(655_360, 8, 16), (8_000_064, 8, 8), (133_321, 2, 8), (2_100, 1, 8), (9, 1, 1), (262_147, 4, 8)]


@pytest.mark.parametrize("N,n_dp,align", CASES)
def test_accumulation_overwrite_then_add(zlib, cuda_device, N, n_dp, align):
    """Over whole shards (one launch) and over a range cutting shards, first
    overwriting and then adding."""
    zb = zlib
    L = zb.zero_layout([N], n_dp, align=align)
    S, P = L.shard, L.padded_n
    A = torch.empty(P, device="cuda")
    Ac = torch.empty(P, device="cuda")
    lo, hi = min(P, S // 2 + 16), max(min(P, S // 2 + 16), P - 5)       # cuts the first and last shard
    ref = None
    for k in range(2):
        g = inputs.grads_bf16(n_dp, N, P, seed=21 + n_dp, step=1, micro=k, outlier_p=0.01)
        qg, q_ref, s_ref = _quantize(zb, L, g)
        qs, ss = qg.sources()
        zb.zero_accumulate_int8(L, qs, ss, BLOCK, A, 0, 0, P, k == 0)
        zb.zero_accumulate_int8(L, qs, ss, BLOCK, Ac, 0, lo, hi, k == 0)
        torch.cuda.synchronize()
        ref = oracle.accumulate_reduce_int8(ref, q_ref, s_ref, n_dp, BLOCK, k == 0)
        parity.assert_bit_exact_f32(A, ref)
        parity.assert_bit_exact_f32(Ac[lo:hi], ref[lo:hi])


@pytest.mark.parametrize("N,n_dp,align", CASES)
def test_update_whole_shards_and_buckets(zlib, cuda_device, N, n_dp, align):
    """Two steps of the update from 8-bit gradients, bucketed so that buckets
    cut shards (one launch per owner) and over whole shards (one launch)."""
    zb = zlib
    for bucket in (max(8, (N // 3) // 8 * 8), 500_000_000):
        L = zb.zero_layout([N], n_dp, align=align, bucket_elems=bucket)
        P = L.padded_n
        w0 = inputs.master_weights(N, P, seed=n_dp + 3)
        st = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
        out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
        ref = [parity.f32(w0), np.zeros(P, np.float32), np.zeros(P, np.float32)]
        for t in (1, 2):
            g = inputs.grads_bf16(n_dp, N, P, seed=n_dp + 3, step=t, outlier_p=0.01)
            qg, q_ref, s_ref = _quantize(zb, L, g)
            zstep.zero12_step_int8(L, qg, *st, out, _hp(zb, t))
            torch.cuda.synchronize()
            out_ref, *ref = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_dp, BLOCK, n_dp, *ref, HP, t)
            parity.assert_state(st, ref, what=f"bucket={bucket} t={t} ")
            assert np.array_equal(parity.bits(out), out_ref)


@pytest.mark.parametrize("n_src", [1, 2, 4, 8])
def test_every_staged_source_count(zlib, cuda_device, n_src):
    """The accumulation and the update with 1, 2, 4 and 8 sources on aligned
    slices of several tiles."""
    zb = zlib
    N = 40_960 * n_src + 37
    L = zb.zero_layout([N], n_src, align=16)
    P = L.padded_n
    g = inputs.grads_bf16(n_src, N, P, seed=40 + n_src, step=1)
    qg, q_ref, s_ref = _quantize(zb, L, g)
    qs, ss = qg.sources()
    A = torch.empty(P, device="cuda")
    zb.zero_accumulate_int8(L, qs, ss, BLOCK, A, 0, 0, P, True)
    w0 = inputs.master_weights(N, P, seed=41)
    st = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    zb.zero_reduce_scatter_adamw_int8(L, qs, ss, BLOCK, float(n_src), 0, n_src, 0, P, *st, out,
                                      zb.ZERO_OUT_FULL, _hp(zb, 1))
    torch.cuda.synchronize()
    parity.assert_bit_exact_f32(A, oracle.accumulate_reduce_int8(None, q_ref, s_ref, n_src, BLOCK, True))
    out_ref, *ref = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_src, BLOCK, n_src, parity.f32(w0),
                                                    np.zeros(P, np.float32), np.zeros(P, np.float32), HP, 1)
    parity.assert_state(st, ref)
    assert np.array_equal(parity.bits(out), out_ref)


@pytest.mark.parametrize("numels,n_dp", [([655_360], 8), ([1_000_000, 24], 4), ([2_048], 2)])
def test_update_with_8bit_output(zlib, cuda_device, numels, n_dp):
    """From the ranks' 8-bit gradients to the owners' 8-bit shards over whole
    256-element-aligned shards: codes and scales equal the update into bf16
    followed by the oracle's quantizer."""
    zb = zlib
    L = zb.zero_layout(numels, n_dp, align=256)
    P, S = L.padded_n, L.shard
    N = L.n
    w0 = inputs.master_weights(N, P, seed=7)
    st = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    q_out = torch.zeros(P, dtype=torch.int8, device="cuda")
    s_out = torch.zeros(P // 256, device="cuda")
    g = inputs.grads_bf16(n_dp, N, P, seed=8, step=1, outlier_p=0.01)
    qg, q_ref, s_ref = _quantize(zb, L, g)
    qs, ss = qg.sources()
    zb.zero_reduce_scatter_adamw_int8_q8(L, qs, ss, BLOCK, float(n_dp), 0, n_dp, 0, P, *st, q_out, s_out,
                                         256, _hp(zb, 1))
    torch.cuda.synchronize()
    out_ref, *ref = oracle.qgrad_rs_adamw_reference(q_ref, s_ref, n_dp, BLOCK, n_dp, parity.f32(w0),
                                                    np.zeros(P, np.float32), np.zeros(P, np.float32), HP, 1)
    parity.assert_state(st, ref)
    for o in range(n_dp):
        qo, so = oracle.quantize_int8(out_ref[o * S:(o + 1) * S], 256)
        np.testing.assert_array_equal(q_out[o * S:(o + 1) * S].cpu().numpy(), qo)
        np.testing.assert_array_equal(s_out[o * S // 256:(o + 1) * S // 256].cpu().numpy(), so)


@pytest.mark.skipif(bool(os.environ.get("ZGB_TEST_LIB")), reason="already running against a variant")
def test_staged_build_matches_the_oracle(tmp_path, cuda_device):
    from zero_sharded_mixed_gb300 import build as zbuild
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib = zbuild.build(defines=["ZGB_QWS=3"], out=str(tmp_path / "libzero_gb300_qws.so"))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.abspath(__file__)], cwd=root, env=dict(os.environ, ZGB_TEST_LIB=lib),
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
