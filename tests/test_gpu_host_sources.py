"""Gradient sources in pinned host memory: the fused update reads them over the
host link itself (zero_reduce_scatter_adamw accepts pinned, mapped host
pointers as sources).  The result is bit-identical to device sources and to the
oracle; pageable host memory is refused."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

HP = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


def _hp(zb, t):
    return zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, t)


@pytest.mark.parametrize("N,n_dp,bucket", [(300_007, 4, 100_000), (65_541, 8, 500_000_000),
                                           (4097, 3, 1000)])
def test_pinned_host_sources_match_device_sources_and_oracle(zlib, cuda_device, N, n_dp, bucket):
    zb = zlib
    L = zb.zero_layout([N], n_dp, bucket_elems=bucket)
    P = L.padded_n
    w0 = inputs.master_weights(N, P, seed=n_dp)
    st_h = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    st_d = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    out_h = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    out_d = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    host_out = torch.empty(P, dtype=torch.bfloat16, pin_memory=True)
    pipe = zstep.HostDirect(L)
    ref = [parity.f32(w0), np.zeros(P, np.float32), np.zeros(P, np.float32)]
    for t in (1, 2):
        g = inputs.grads_bf16(n_dp, N, P, seed=n_dp, step=t)
        g_host = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
        g_host.copy_(g)
        pipe.step(g_host, *st_h, out_h, host_out, _hp(zb, t))
        zstep.zero12_step(L, [g[r].cuda() for r in range(n_dp)], *st_d, out_d, _hp(zb, t))
        torch.cuda.synchronize()
        out_ref, *ref = oracle.rs_adamw_reference(parity.bits(g), n_dp, *ref, HP, t)
        parity.assert_state(st_h, ref, what=f"t={t} ")
        for a, b in zip(st_h, st_d):
            parity.assert_bit_exact_f32(a, parity.f32(b))
        assert np.array_equal(parity.bits(host_out), out_ref)
        assert np.array_equal(parity.bits(out_d), out_ref)


def test_pageable_host_sources_are_refused(zlib, cuda_device):
    zb = zlib
    L = zb.zero_layout([4096], 2)
    P = L.padded_n
    g = torch.zeros((2, P), dtype=torch.bfloat16)                  # pageable
    st = [torch.zeros(P, device="cuda") for _ in range(3)]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        zb.zero_reduce_scatter_adamw(L, [g[0], g[1]], zb.ZERO_BF16, 0, 2.0, 0, 2, 0, P, *st, out,
                                     zb.ZERO_OUT_FULL, _hp(zb, 1))
    srcs = (ctypes.c_void_p * 2)(g[0].data_ptr(), g[1].data_ptr())
    hp = _hp(zb, 1)
    rc = zb.load().zero_reduce_scatter_adamw(ctypes.byref(L), srcs, 2, zb.ZERO_BF16, 0, 2.0, 0, 2, 0, P,
                                             *[x.data_ptr() for x in st], out.data_ptr(),
                                             zb.ZERO_OUT_FULL, ctypes.byref(hp), None)
    assert rc == -1
    # the state must still be device memory, even when pinned
    w_pinned = torch.zeros(P, pin_memory=True)
    gd = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(ValueError):
        zb.zero_reduce_scatter_adamw(L, gd, zb.ZERO_BF16, 0, 2.0, 0, 2, 0, P, w_pinned, st[1], st[2],
                                     out, zb.ZERO_OUT_FULL, _hp(zb, 1))
    zb.zero_status_check()


@pytest.mark.parametrize("defer_out", [False, True])
@pytest.mark.parametrize("N,n_dp,bucket,chunk", [(300_007, 4, 100_000, None), (65_541, 8, 20_000, 7_000)])
def test_copy_pipeline_matches_the_oracle(zlib, cuda_device, N, n_dp, bucket, chunk, defer_out):
    """The e2e pipeline (gradients copied from pinned host memory bucket by
    bucket, each bucket updated once its copies land, the bf16 result copied
    back to pinned host memory, overlapped or after the last gradient copy):
    the state and the host result equal the oracle's, three steps."""
    zb = zlib
    L = zb.zero_layout([N], n_dp, bucket_elems=bucket)
    P = L.padded_n
    w0 = inputs.master_weights(N, P, seed=n_dp + 1)
    st = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    dev_g = torch.empty((n_dp, P), dtype=torch.bfloat16, device="cuda")
    host_out = torch.empty(P, dtype=torch.bfloat16, pin_memory=True)
    pipe = zstep.HostPipeline(L, chunk_elems=chunk, defer_out=defer_out)
    ref = [parity.f32(w0), np.zeros(P, np.float32), np.zeros(P, np.float32)]
    for t in (1, 2, 3):
        g = inputs.grads_bf16(n_dp, N, P, seed=n_dp + 1, step=t)
        g_host = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
        g_host.copy_(g)
        pipe.step(g_host, dev_g, *st, out, host_out, _hp(zb, t))
        torch.cuda.synchronize()
        out_ref, *ref = oracle.rs_adamw_reference(parity.bits(g), n_dp, *ref, HP, t)
        parity.assert_state(st, ref, what=f"t={t} ")
        assert np.array_equal(parity.bits(host_out), out_ref)
        assert torch.equal(dev_g.cpu().view(torch.int16), g.view(torch.int16))


def test_copy_pipeline_from_one_shared_host_row(zlib, cuda_device):
    """The e2e pipeline fed by one pinned host row that every simulated rank's
    copy reads (a stride-0 view; the benchmark's fallback when the host cannot
    pin every rank's gradients): every device row receives that row, and the
    step equals the oracle's with all ranks holding it."""
    zb = zlib
    N, n_dp, bucket = 200_003, 8, 60_000
    L = zb.zero_layout([N], n_dp, bucket_elems=bucket)
    P = L.padded_n
    w0 = inputs.master_weights(N, P, seed=11)
    st = [w0.cuda(), torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    dev_g = torch.empty((n_dp, P), dtype=torch.bfloat16, device="cuda")
    host_out = torch.empty(P, dtype=torch.bfloat16, pin_memory=True)
    g = inputs.grads_bf16(1, N, P, seed=12, step=1)
    row = torch.empty(P, dtype=torch.bfloat16, pin_memory=True)
    row.copy_(g[0])
    shared = row.expand(n_dp, P)
    assert shared.is_pinned() and shared.stride(0) == 0
    zstep.HostPipeline(L).step(shared, dev_g, *st, out, host_out, _hp(zb, 1))
    torch.cuda.synchronize()
    rows = np.repeat(parity.bits(g), n_dp, axis=0)
    assert np.array_equal(dev_g.cpu().view(torch.int16).numpy().view(np.uint16), rows)
    out_ref, *ref = oracle.rs_adamw_reference(rows, n_dp, parity.f32(w0), np.zeros(P, np.float32),
                                              np.zeros(P, np.float32), HP, 1)
    parity.assert_state(st, ref)
    assert np.array_equal(parity.bits(host_out), out_ref)
