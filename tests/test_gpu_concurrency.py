"""Two host threads, each driving its own ZeRO problem on its own CUDA stream
through the library at the same time: the results equal those of running the
two problems one after the other (the library keeps no per-call state)."""
import threading

import pytest
import torch

from tests import parity
from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu


def _problem(zb, N, n_dp, seed, bucket):
    L = zb.zero_layout([N], n_dp, bucket_elems=bucket)
    P = L.padded_n
    grads = [inputs.grads_bf16(n_dp, N, P, seed=seed, step=t).cuda() for t in (1, 2, 3)]
    w = inputs.master_weights(N, P, seed=seed).cuda()
    return L, grads, w


def _run(zb, L, grads, w0, stream, out_list):
    with torch.cuda.stream(stream):
        st = [w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0)]
        out = torch.zeros(L.padded_n, dtype=torch.bfloat16, device="cuda")
        for t, g in enumerate(grads, start=1):
            zstep.zero12_step(L, [g[r] for r in range(L.n_dp)], *st, out, zb.ZeroAdamW.make(step=t),
                              stream=stream)
        stream.synchronize()
    out_list.append((st, out))


def test_two_threads_two_streams(zlib, cuda_device):
    zb = zlib
    pa = _problem(zb, 3_000_017, 4, 1, 1_000_000)
    pb = _problem(zb, 2_000_003, 8, 2, 700_000)
    torch.cuda.synchronize()
    seq_a, seq_b = [], []
    s0 = torch.cuda.Stream()
    _run(zb, *pa, s0, seq_a)
    _run(zb, *pb, s0, seq_b)
    con_a, con_b = [], []
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    ta = threading.Thread(target=_run, args=(zb, *pa, sa, con_a))
    tb = threading.Thread(target=_run, args=(zb, *pb, sb, con_b))
    ta.start(); tb.start(); ta.join(); tb.join()
    torch.cuda.synchronize()
    for (s1, o1), (s2, o2) in ((seq_a[0], con_a[0]), (seq_b[0], con_b[0])):
        for x, y in zip(s1, s2):
            parity.assert_bit_exact_f32(x, y)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
