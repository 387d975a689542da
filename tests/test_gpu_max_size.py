"""Launches whose element indexes pass 2^31 and 2^32.

One flat vector of N = 2^32 + 2^20 + 5 elements at n_dp = 2 (so each shard is
longer than 2^31 and the padded vector longer than 2^32, with a ragged end):
the fused update, the REDUCE accumulation and the gather each run as one
launch over the whole vector, and the 8-bit gradient path (per-rank
quantization, then the update from the codes) as one launch per owner over a
shard of more than 2^31 elements.  Every result is compared with the oracle,
bit for bit, on slices at the start, around 2^31 and 2^32, at the owners'
boundary and at the end with its padding.  About 95 GB on the device."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from zero_sharded_mixed_gb300 import inputs

pytestmark = pytest.mark.gpu

N = 2 ** 32 + 2 ** 20 + 5
N_DP = 2
BLOCK = 256
HP = oracle.AdamW(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
NEED_BYTES = 100 * 10 ** 9


def _slices(S, P):
    """Sample ranges [a, b): each lies in one owner's slice and starts on that
    slice's 256-element block grid, so the 8-bit blocks can be re-derived."""
    def aligned(o, x):
        return o * S + ((x - o * S) // BLOCK) * BLOCK
    return [
        (0, 4096),
        (aligned(0, 2 ** 31 - 2048), aligned(0, 2 ** 31 - 2048) + 4096),   # crosses 2^31
        (aligned(0, S - 4096), S),                                        # owner 0's ragged end
        (S, S + 4096),                                                    # owner 1's start
        (aligned(1, 2 ** 32 - 2048), aligned(1, 2 ** 32 - 2048) + 4096),  # crosses 2^32
        (aligned(1, P - 4096), P),                                        # N and the padding
    ]


@pytest.fixture(scope="module")
def big(zlib, cuda_device):
    free, _ = torch.cuda.mem_get_info()
    if free < NEED_BYTES:
        pytest.skip(f"needs {NEED_BYTES / 1e9:.0f} GB free on the device, {free / 1e9:.0f} GB free")
    zb = zlib
    L = zb.zero_layout([N], N_DP, align=8)
    S, P = L.shard, L.padded_n
    assert S > 2 ** 31 and P > 2 ** 32 and S % BLOCK != 0
    g = torch.empty((N_DP, P), dtype=torch.bfloat16, device="cuda")
    for r in range(N_DP):
        inputs.grad_bf16_into(g[r], N, seed=31, step=1, rank=r)
    state = {"L": L, "g": g, "slices": _slices(S, P)}
    yield state
    state.clear()
    torch.cuda.empty_cache()


def _fresh_state(P):
    w = inputs.master_weights(N, P, seed=32, device="cuda")
    return w, torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")


def test_fused_update_reduce_and_gather(zlib, big):
    zb = zlib
    L, g = big["L"], big["g"]
    S, P = L.shard, L.padded_n
    rows = [g[r] for r in range(N_DP)]
    w, m, v = _fresh_state(P)
    w0 = {ab: parity.f32(w[ab[0]:ab[1]]) for ab in big["slices"]}
    out = torch.empty(P, dtype=torch.bfloat16, device="cuda")
    hp = zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, 1)
    zb.zero_reduce_scatter_adamw(L, rows, zb.ZERO_BF16, 0, float(N_DP), 0, N_DP, 0, P, w, m, v, out,
                                 zb.ZERO_OUT_FULL, hp)
    full = torch.empty(P, dtype=torch.bfloat16, device="cuda")
    zb.zero_gather_layer(L, [out[:S], out[S:]], full)
    torch.cuda.synchronize()
    for a, b in big["slices"]:
        src = parity.bits(g[:, a:b])
        n = b - a
        out_ref, *st = oracle.rs_adamw_reference(src, N_DP, w0[(a, b)], np.zeros(n, np.float32),
                                                 np.zeros(n, np.float32), HP, 1)
        what = f"[{a}, {b}) "
        parity.assert_state([w[a:b], m[a:b], v[a:b]], st, what=what)
        assert np.array_equal(parity.bits(out[a:b]), out_ref), what + "bf16 output"
        assert np.array_equal(parity.bits(full[a:b]), out_ref), what + "gather"
    del full, out
    # REDUCE accumulation over the whole vector, into m
    zb.zero_accumulate(L, zb.ZERO_ACC_REDUCE, rows, zb.ZERO_BF16, 0, m, 0, 0, P, True)
    torch.cuda.synchronize()
    for a, b in big["slices"]:
        ref = oracle.accumulate_reduce(None, parity.bits(g[:, a:b]), True)
        parity.assert_bit_exact_f32(m[a:b], ref, what=f"accumulation [{a}, {b})")
    zb.zero_status_check()


def test_int8_gradient_update(zlib, big):
    zb = zlib
    L, g = big["L"], big["g"]
    S, P = L.shard, L.padded_n
    nb = -(-S // BLOCK)
    q = torch.empty((N_DP, P), dtype=torch.int8, device="cuda")
    sc = torch.empty((N_DP, N_DP * nb), dtype=torch.float32, device="cuda")
    for r in range(N_DP):
        zb.zero_quantize_int8(L, g[r], q[r], sc[r], BLOCK)
    w, m, v = _fresh_state(P)
    w0 = {ab: parity.f32(w[ab[0]:ab[1]]) for ab in big["slices"]}
    out = torch.empty(P, dtype=torch.bfloat16, device="cuda")
    hp = zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, 1)
    zb.zero_reduce_scatter_adamw_int8(L, [q[r] for r in range(N_DP)], [sc[r] for r in range(N_DP)],
                                      BLOCK, float(N_DP), 0, N_DP, 0, P, w, m, v, out,
                                      zb.ZERO_OUT_FULL, hp)
    torch.cuda.synchronize()
    for a, b in big["slices"]:
        o = a // S
        k0 = (a - o * S) // BLOCK
        k1 = k0 + -(-(b - a) // BLOCK)
        what = f"[{a}, {b}) "
        qs = q[:, a:b].cpu().numpy()
        ss = sc[:, o * nb + k0:o * nb + k1].cpu().numpy()
        for r in range(N_DP):
            q_ref, s_ref = oracle.quantize_int8(parity.bits(g[r, a:b]), BLOCK)
            assert np.array_equal(qs[r], q_ref), what + f"codes of rank {r}"
            assert np.array_equal(ss[r].view(np.uint32), s_ref.view(np.uint32)), what + f"scales of rank {r}"
        n = b - a
        out_ref, *st = oracle.qgrad_rs_adamw_reference(qs, ss, 1, BLOCK, N_DP, w0[(a, b)],
                                                       np.zeros(n, np.float32), np.zeros(n, np.float32),
                                                       HP, 1)
        parity.assert_state([w[a:b], m[a:b], v[a:b]], st, what=what)
        assert np.array_equal(parity.bits(out[a:b]), out_ref), what + "bf16 output"
    zb.zero_status_check()


def test_int8_gradient_update_over_a_range_cutting_a_shard(zlib, big):
    """The 8-bit update over [lo, P) with lo inside owner 0's slice: one stream
    over a range longer than 2^32 that crosses the owner boundary at S > 2^31,
    each vector finding its owner.  Elements before lo stay untouched."""
    zb = zlib
    L, g = big["L"], big["g"]
    S, P = L.shard, L.padded_n
    nb = -(-S // BLOCK)
    q = torch.empty((N_DP, P), dtype=torch.int8, device="cuda")
    sc = torch.empty((N_DP, N_DP * nb), dtype=torch.float32, device="cuda")
    for r in range(N_DP):
        zb.zero_quantize_int8(L, g[r], q[r], sc[r], BLOCK)
    lo = (2 ** 30 // BLOCK) * BLOCK + 8 * 37           # on the vector grid, off the block grid
    w, m, v = _fresh_state(P)
    slices = [(a, b) for a, b in big["slices"] if a >= lo] + [(lo, lo + 4096)]
    w0 = {ab: parity.f32(w[ab[0]:ab[1]]) for ab in slices + [(lo - 64, lo)]}
    out = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    hp = zb.ZeroAdamW.make(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, 1)
    zb.zero_reduce_scatter_adamw_int8(L, [q[r] for r in range(N_DP)], [sc[r] for r in range(N_DP)],
                                      BLOCK, float(N_DP), 0, N_DP, lo, P, w, m, v, out,
                                      zb.ZERO_OUT_FULL, hp)
    torch.cuda.synchronize()
    for a, b in slices:
        o = a // S
        k0 = (a - o * S) // BLOCK
        k1 = -(-(b - o * S) // BLOCK)
        off = (a - o * S) - k0 * BLOCK                   # the slice's offset inside its first block
        qs = q[:, a - off:b].cpu().numpy()
        ss = sc[:, o * nb + k0:o * nb + k1].cpu().numpy()
        n = b - a
        out_ref, *st = oracle.qgrad_rs_adamw_reference(qs, ss, 1, BLOCK, N_DP, np.concatenate(
            [np.zeros(off, np.float32), w0[(a, b)]]), np.zeros(n + off, np.float32),
            np.zeros(n + off, np.float32), HP, 1)
        what = f"[{a}, {b}) "
        parity.assert_state([w[a:b], m[a:b], v[a:b]], [x[off:] for x in st], what=what)
        assert np.array_equal(parity.bits(out[a:b]), out_ref[off:]), what + "bf16 output"
    parity.assert_bit_exact_f32(w[lo - 64:lo], w0[(lo - 64, lo)], what="before the range")
    assert not m[lo - 64:lo].any() and not out[lo - 64:lo].view(torch.int16).any()
    zb.zero_status_check()


def test_cast_of_the_whole_vector(zlib, big):
    """The library's bf16 cast over P > 2^32 elements, sampled slices bit for
    bit against the oracle's cast."""
    zb = zlib
    P = big["L"].padded_n
    w, _, _ = _fresh_state(P)
    out = torch.empty(P, dtype=torch.bfloat16, device="cuda")
    zb.zero_cast_bf16(w, out)
    torch.cuda.synchronize()
    for a, b in big["slices"]:
        assert np.array_equal(parity.bits(out[a:b]), oracle.cast_bf16(parity.f32(w[a:b]))), f"[{a}, {b})"
    zb.zero_status_check()
