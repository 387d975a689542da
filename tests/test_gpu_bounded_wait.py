"""Failure detection without a GPU fault: a kernel waits on an mbarrier that
nothing completes, with a bound of about a millisecond.  The wait gives up,
the kernel records ZERO_ETIMEOUT and returns; zero_status_check reports it
once, and the context keeps running ordinary work."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable(zlib, cuda_device):
    zb = zlib
    zb.zero_status_check()                                    # nothing pending
    zb.zero_selftest_bounded_wait(2_000_000)                  # ~1 ms of SM clock
    with pytest.raises(zb.ZeroError) as e:
        zb.zero_status_check()
    assert e.value.code == zb.ZERO_ETIMEOUT
    zb.zero_status_check()                                    # reported once, then cleared
    # ordinary work still runs and is right
    N, n_dp = 100_000, 2
    L = zb.zero_layout([N], n_dp)
    g = inputs.grads_bf16(n_dp, N, L.padded_n, seed=1, step=1)
    w0 = inputs.master_weights(N, L.padded_n, seed=1)
    st = [w0.cuda(), torch.zeros(L.padded_n, device="cuda"), torch.zeros(L.padded_n, device="cuda")]
    out = torch.zeros(L.padded_n, dtype=torch.bfloat16, device="cuda")
    zb.zero_reduce_scatter_adamw(L, [g[r].cuda() for r in range(n_dp)], zb.ZERO_BF16, 0, 2.0, 0, n_dp,
                                 0, L.padded_n, *st, out, zb.ZERO_OUT_FULL, zb.ZeroAdamW.make(step=1))
    zb.zero_status_check()
    z = np.zeros(L.padded_n, np.float32)
    ref_out, *ref = oracle.rs_adamw_reference(parity.bits(g), n_dp, parity.f32(w0), z, z, oracle.AdamW(), 1)
    parity.assert_state(st, ref)
    assert np.array_equal(parity.bits(out), ref_out)


def test_selftest_rejects_out_of_range_limits(zlib, cuda_device):
    zb = zlib
    for bad in (0, -5, 1 << 40):
        with pytest.raises(zb.ZeroError):
            zb.zero_selftest_bounded_wait(bad)
