"""Guard bands around every buffer of every entry point.

Each buffer a call touches is the middle of a larger allocation whose two
guard bands (16 KiB each) are filled with random bytes.  After the call:
- every guard band is byte for byte what it was, so nothing wrote out of bounds;
- every input (gradients, accumulators, shards, codes, scales) is byte for byte
  what it was, since the calls read their sources only.
Each case runs on the vector kernels (16-byte aligned, sizes on the 8-element
grid) and, with buffers shifted off the grid, on the element kernels, at
ragged sizes.  This is the check that an out-of-bounds store would fail; it
needs no sanitizer."""
import pytest
import torch

from zero_sharded_mixed_gb300 import inputs
from zero_sharded_mixed_gb300 import step as zstep

pytestmark = pytest.mark.gpu

GUARD_BYTES = 16384


class Guarded:
    """A length-n tensor of `dtype` in the middle of a guarded allocation; the
    tensor starts `shift` elements after the guard (shift 1 moves a 2- or
    4-byte type off the 16-byte grid)."""

    _seed = 0

    def __init__(self, n, dtype, shift=0, data=None):
        es = torch.empty(0, dtype=dtype).element_size()
        g = GUARD_BYTES // es
        self.lo, self.hi = g + shift, g + shift + n
        self.buf = torch.empty(self.hi + g, dtype=dtype, device="cuda")
        Guarded._seed += 1
        gen = torch.Generator(device="cuda").manual_seed(1000 + Guarded._seed)
        self.buf.view(torch.uint8).random_(0, 256, generator=gen)
        self.t = self.buf[self.lo:self.hi]
        if data is not None:
            self.t.copy_(data)
        self.snap = self.buf.clone()

    def guards_intact(self):
        b = self.buf.view(torch.uint8)
        s = self.snap.view(torch.uint8)
        es = self.buf.element_size()
        return bool(torch.equal(b[:self.lo * es], s[:self.lo * es]) and
                    torch.equal(b[self.hi * es:], s[self.hi * es:]))

    def unchanged(self):
        return bool(torch.equal(self.buf.view(torch.uint8), self.snap.view(torch.uint8)))


def _check(outputs, inputs_):
    torch.cuda.synchronize()
    for name, g in outputs.items():
        assert g.guards_intact(), f"{name}: a guard band was written"
    for name, g in inputs_.items():
        assert g.unchanged(), f"{name}: an input was modified"


def _grads(n_src, n, shift, dtype=torch.bfloat16, seed=1):
    g = inputs.grads_bf16(n_src, n, n, seed=seed, step=1).to(dtype)
    return [Guarded(n, dtype, shift, g[r].cuda()) for r in range(n_src)]


def _state(n, shift):
    w = inputs.master_weights(n, n, seed=2).cuda()
    return (Guarded(n, torch.float32, shift, w), Guarded(n, torch.float32, shift, torch.zeros(n)),
            Guarded(n, torch.float32, shift, torch.zeros(n)))


@pytest.mark.parametrize("align,shift", [(8, 0), (1, 1)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_fused_update(zlib, cuda_device, align, shift, dtype):
    """Owners 1..2 of 4, buckets crossing owners, sources read from src_base = S,
    both output modes; and the clipped update with its norm pass."""
    zb = zlib
    N, n_dp = 20_011, 4
    L = zb.zero_layout([N], n_dp, align=align, bucket_elems=3001)
    S, P = L.shard, L.padded_n
    lo, hi = S, 3 * S
    src = _grads(n_dp, hi - lo, shift, dtype)
    w, m, v = _state(hi - lo, shift)
    out_full = Guarded(P, torch.bfloat16, shift)
    out_shard = Guarded(hi - lo, torch.bfloat16, shift)
    dt = zb.ZERO_BF16 if dtype == torch.bfloat16 else zb.ZERO_F32
    hp = zb.ZeroAdamW.make(step=1)
    rows = [g.t for g in src]
    for s, e in zstep.bucket_ranges(L, lo, hi):
        zb.zero_reduce_scatter_adamw(L, rows, dt, lo, float(n_dp), 1, 3, s, e, w.t, m.t, v.t,
                                     out_full.t, zb.ZERO_OUT_FULL, hp)
        zb.zero_reduce_scatter_adamw(L, rows, dt, lo, float(n_dp), 1, 3, s, e, w.t, m.t, v.t,
                                     out_shard.t, zb.ZERO_OUT_SHARD, hp)
    ws = Guarded(zb.zero_grad_norm_workspace() // 8, torch.float64)
    nsq = Guarded(1, torch.float64)
    for j, (s, e) in enumerate(zstep.bucket_ranges(L, lo, hi)):
        zb.zero_grad_norm_sq(L, rows, dt, lo, float(n_dp), s, e, ws.t, nsq.t, j > 0)
    for s, e in zstep.bucket_ranges(L, lo, hi):
        zb.zero_reduce_scatter_adamw_clip(L, rows, dt, lo, float(n_dp), 1, 3, s, e, w.t, m.t, v.t,
                                          out_full.t, zb.ZERO_OUT_FULL, hp, nsq.t, 0.5)
    _check({"w": w, "m": m, "v": v, "out_full": out_full, "out_shard": out_shard, "workspace": ws,
            "norm_sq": nsq}, {f"src[{r}]": g for r, g in enumerate(src)})


@pytest.mark.parametrize("align,shift", [(8, 0), (1, 1)])
def test_accumulation_and_fused_finish(zlib, cuda_device, align, shift):
    zb = zlib
    N, n_dp = 10_005, 3
    L = zb.zero_layout([N], n_dp, align=align, bucket_elems=2003)
    P = L.padded_n
    src = _grads(n_dp, P, shift)
    rows = [g.t for g in src]
    acc = [Guarded(P, torch.float32, shift, torch.zeros(P)) for _ in range(n_dp)]
    A = Guarded(P, torch.float32, shift, torch.zeros(P))
    for first in (True, False):
        for r in range(n_dp):
            zb.zero_accumulate(L, zb.ZERO_ACC_LOCAL, [rows[r]], zb.ZERO_BF16, 0, acc[r].t, 0, 0, P, first)
        zb.zero_accumulate(L, zb.ZERO_ACC_REDUCE, rows, zb.ZERO_BF16, 0, A.t, 0, 0, P, first)
    acc_in = [Guarded(P, torch.float32, shift, a.t) for a in acc]
    A_in = Guarded(P, torch.float32, shift, A.t)
    w, m, v = _state(P, shift)
    out = Guarded(P, torch.bfloat16, shift)
    hp = zb.ZeroAdamW.make(step=1)
    for s, e in zstep.bucket_ranges(L):
        zb.zero_accumulate_adamw(L, zb.ZERO_ACC_LOCAL, [a.t for a in acc_in], 0, rows, 0, 3.0 * n_dp,
                                 0, n_dp, s, e, w.t, m.t, v.t, out.t, zb.ZERO_OUT_FULL, hp)
        zb.zero_accumulate_adamw(L, zb.ZERO_ACC_REDUCE, [A_in.t], 0, rows, 0, 3.0 * n_dp,
                                 0, n_dp, s, e, w.t, m.t, v.t, out.t, zb.ZERO_OUT_FULL, hp)
    _check({**{f"acc[{r}]": a for r, a in enumerate(acc)}, "A": A, "w": w, "m": m, "v": v, "out": out},
           {**{f"src[{r}]": g for r, g in enumerate(src)},
            **{f"acc_in[{r}]": a for r, a in enumerate(acc_in)}, "A_in": A_in})


@pytest.mark.parametrize("align,shift,block", [(8, 0, 256), (8, 0, 1024), (1, 1, 512)])
def test_gathers_and_8bit_paths(zlib, cuda_device, align, shift, block):
    """The stage-3 gather, the 8-bit weight quantizer and gather, and the 8-bit
    gradient update and accumulation."""
    zb = zlib
    N, n_dp = 30_011, 5
    L = zb.zero_layout([N], n_dp, align=align, bucket_elems=7001)
    S, P = L.shard, L.padded_n
    nb = -(-S // block)
    w0 = inputs.master_weights(N, P, seed=3).to(torch.bfloat16)
    shards = [Guarded(S, torch.bfloat16, shift, w0[o * S:(o + 1) * S].cuda()) for o in range(n_dp)]
    full = Guarded(P, torch.bfloat16, shift)
    zb.zero_gather_layer(L, [s.t for s in shards], full.t)
    packed = Guarded(P, torch.bfloat16, shift, w0.cuda())
    q = Guarded(P, torch.int8, shift)
    sc = Guarded(n_dp * nb, torch.float32, shift)
    zb.zero_quantize_int8(L, packed.t, q.t, sc.t, block)
    torch.cuda.synchronize()
    q_in = [Guarded(S, torch.int8, shift, q.t[o * S:(o + 1) * S]) for o in range(n_dp)]
    s_in = [Guarded(nb, torch.float32, shift, sc.t[o * nb:(o + 1) * nb]) for o in range(n_dp)]
    full8 = Guarded(P, torch.bfloat16, shift)
    zb.zero_gather_layer_int8(L, [x.t for x in q_in], [x.t for x in s_in], full8.t, block)
    # 8-bit gradients: each rank's whole gradient quantized, then the owners' update and accumulation
    g = inputs.grads_bf16(n_dp, N, P, seed=4, step=1)
    g_in = [Guarded(P, torch.bfloat16, shift, g[r].cuda()) for r in range(n_dp)]
    qg = [Guarded(P, torch.int8, shift) for _ in range(n_dp)]
    sg = [Guarded(n_dp * nb, torch.float32, shift) for _ in range(n_dp)]
    for r in range(n_dp):
        zb.zero_quantize_int8(L, g_in[r].t, qg[r].t, sg[r].t, block)
    torch.cuda.synchronize()
    qg_in = [Guarded(P, torch.int8, shift, x.t) for x in qg]
    sg_in = [Guarded(n_dp * nb, torch.float32, shift, x.t) for x in sg]
    w, m, v = _state(P, shift)
    out = Guarded(P, torch.bfloat16, shift)
    hp = zb.ZeroAdamW.make(step=1)
    for s, e in zstep.bucket_ranges(L):
        zb.zero_reduce_scatter_adamw_int8(L, [x.t for x in qg_in], [x.t for x in sg_in], block,
                                          float(n_dp), 0, n_dp, s, e, w.t, m.t, v.t, out.t,
                                          zb.ZERO_OUT_FULL, hp)
    A = Guarded(P, torch.float32, shift)
    Ao = Guarded(S, torch.float32, shift)
    for first in (True, False):
        zb.zero_accumulate_int8(L, [x.t for x in qg_in], [x.t for x in sg_in], block, A.t, 0, 0, P, first)
        zb.zero_accumulate_int8(L, [x.t for x in qg_in], [x.t for x in sg_in], block, Ao.t, 2 * S,
                                2 * S, 3 * S, first)
    _check({"full": full, "q": q, "scales": sc, "full8": full8, "w": w, "m": m, "v": v, "out": out,
            "A": A, "A_owner2": Ao, **{f"qg[{r}]": x for r, x in enumerate(qg)},
            **{f"sg[{r}]": x for r, x in enumerate(sg)}},
           {**{f"shard[{o}]": s for o, s in enumerate(shards)}, "packed": packed,
            **{f"q_in[{o}]": x for o, x in enumerate(q_in)}, **{f"s_in[{o}]": x for o, x in enumerate(s_in)},
            **{f"g[{r}]": x for r, x in enumerate(g_in)}, **{f"qg_in[{r}]": x for r, x in enumerate(qg_in)},
            **{f"sg_in[{r}]": x for r, x in enumerate(sg_in)}})
    zb.zero_status_check()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_q8_update(zlib, cuda_device, dtype):
    """The update with the 8-bit output, owners 1..3 of 5, a range on block
    boundaries inside them."""
    zb = zlib
    N, n_dp, block = 40_000, 5, 256
    L = zb.zero_layout([N], n_dp, align=block)
    S = L.shard
    lo, hi = S + 2 * block, 4 * S - block
    src = _grads(n_dp, hi - lo, 0, dtype)
    w, m, v = _state(3 * S, 0)
    q = Guarded(3 * S, torch.int8)
    sc = Guarded(3 * S // block, torch.float32)
    dt = zb.ZERO_BF16 if dtype == torch.bfloat16 else zb.ZERO_F32
    zb.zero_reduce_scatter_adamw_q8(L, [g.t for g in src], dt, lo, float(n_dp), 1, 4, lo, hi, w.t, m.t,
                                    v.t, q.t, sc.t, block, zb.ZeroAdamW.make(step=1))
    _check({"w": w, "m": m, "v": v, "q": q, "scales": sc}, {f"src[{r}]": g for r, g in enumerate(src)})


def test_int8_gradient_update_with_8bit_output(zlib, cuda_device):
    zb = zlib
    N, n_dp, block = 40_000, 5, 256
    L = zb.zero_layout([N], n_dp, align=block)
    S, P = L.shard, L.padded_n
    g = inputs.grads_bf16(n_dp, N, P, seed=6, step=1)
    qg = [Guarded(P, torch.int8) for _ in range(n_dp)]
    sg = [Guarded(P // block, torch.float32) for _ in range(n_dp)]
    for r in range(n_dp):
        zb.zero_quantize_int8(L, g[r].cuda(), qg[r].t, sg[r].t, block)
    torch.cuda.synchronize()
    qg_in = [Guarded(P, torch.int8, 0, x.t) for x in qg]
    sg_in = [Guarded(P // block, torch.float32, 0, x.t) for x in sg]
    w, m, v = _state(3 * S, 0)
    q = Guarded(3 * S, torch.int8)
    sc = Guarded(3 * S // block, torch.float32)
    lo, hi = S + block, 4 * S - 2 * block
    zb.zero_reduce_scatter_adamw_int8_q8(L, [x.t for x in qg_in], [x.t for x in sg_in], block, float(n_dp),
                                         1, 4, lo, hi, w.t, m.t, v.t, q.t, sc.t, block,
                                         zb.ZeroAdamW.make(step=1))
    _check({"w": w, "m": m, "v": v, "q": q, "scales": sc},
           {**{f"qg[{r}]": x for r, x in enumerate(qg_in)}, **{f"sg[{r}]": x for r, x in enumerate(sg_in)}})


@pytest.mark.parametrize("shift", [0, 1])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 100_003])
def test_cast(zlib, cuda_device, n, shift):
    """The bf16 cast of master weights: the output's guard bands and the fp32
    source stay untouched, on the vector kernel and off the 16-byte grid."""
    w = Guarded(n, torch.float32, shift, inputs.master_weights(n, n, seed=5).cuda())
    out = Guarded(n, torch.bfloat16, shift)
    zlib.zero_cast_bf16(w.t, out.t)
    _check({"out": out}, {"master": w})
    assert torch.equal(out.t.view(torch.int16), w.t.to(torch.bfloat16).view(torch.int16))
