"""Oracle for the ZeRO stage-1/2/3 sharded mixed-precision step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the ``zero_sharded_mixed_gb300`` package and its CUDA library)
never imports, links or calls anything here, and nothing here imports the
product package.

Two parts:

* ``zero_oracle.c`` -- plain scalar C (built with ``-O2 -ffp-contract=off``):
  layout, reduce-scatter as a mean, fp32 AdamW with bias correction and
  decoupled weight decay, round-to-nearest-even bf16 cast, all-gather, the
  ZeRO-1/2 step over simulated ranks, the plain data-parallel step, and the
  two gradient-accumulation orders.  The numpy wrappers below only marshal
  arrays into it.
* ``formulas.py`` -- the per-GPU model-state bytes and the per-GPU
  communication bytes of each stage ("ZeRO and FSDP", sections "Memory per
  GPU" and "Communication volume").

Every function's pins (what fixes it other than itself) live in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .formulas import zero_comm_bytes, zero_memory  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: every fp32 multiply and add is rounded on its own, as the
# C source is written; gcc would otherwise fuse them on aarch64.
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc), if stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = configure(ctypes.CDLL(build()))
        return _lib


def configure(lib):
    """Declare the C signatures on a loaded oracle library and return it."""
    i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    p = ctypes.c_void_p
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = f32
    lib.oracle_f32_to_bf16.argtypes = [f32]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_cast_bf16.argtypes = [p, p, i64]
    lib.oracle_cast_bf16.restype = None
    lib.oracle_layout.argtypes = [p, i32, i32, i64, i64, p, p]
    lib.oracle_layout.restype = ctypes.c_int
    lib.oracle_reduce_mean_bf16.argtypes = [p, i32, i64, i64, f32, p]
    lib.oracle_reduce_mean_bf16.restype = None
    lib.oracle_reduce_mean_f32.argtypes = [p, i32, i64, i64, f32, p]
    lib.oracle_reduce_mean_f32.restype = None
    lib.oracle_bias_corrections.argtypes = [f32, f32, i64, p, p]
    lib.oracle_bias_corrections.restype = None
    lib.oracle_adamw.argtypes = [p, p, p, p, i64, f32, f32, f32, f32, f32, i64]
    lib.oracle_adamw.restype = None
    lib.oracle_zero_step.argtypes = [p, i32, i64, p, p, p, p, i32,
                                     f32, f32, f32, f32, f32, i64]
    lib.oracle_zero_step.restype = ctypes.c_int
    lib.oracle_dp_step.argtypes = [p, i32, i64, p, p, p, p,
                                   f32, f32, f32, f32, f32, i64]
    lib.oracle_dp_step.restype = ctypes.c_int
    lib.oracle_accumulate_local.argtypes = [p, p, i64, i32]
    lib.oracle_accumulate_local.restype = None
    lib.oracle_accumulate_reduce.argtypes = [p, p, i32, i64, i64, i32]
    lib.oracle_accumulate_reduce.restype = None
    lib.oracle_all_gather_bf16.argtypes = [p, i32, i64, p]
    lib.oracle_all_gather_bf16.restype = None
    lib.oracle_grad_norm_sq_bf16.argtypes = [p, i32, i64, i64, f32]
    lib.oracle_grad_norm_sq_bf16.restype = ctypes.c_double
    lib.oracle_grad_norm_sq_f32.argtypes = [p, i32, i64, i64, f32]
    lib.oracle_grad_norm_sq_f32.restype = ctypes.c_double
    lib.oracle_clip_coef.argtypes = [ctypes.c_double, f32]
    lib.oracle_clip_coef.restype = f32
    lib.oracle_scale.argtypes = [p, i64, f32]
    lib.oracle_scale.restype = None
    lib.oracle_quantize_int8.argtypes = [p, i64, i32, p, p]
    lib.oracle_quantize_int8.restype = None
    lib.oracle_dequantize_int8.argtypes = [p, p, i64, i32, p]
    lib.oracle_dequantize_int8.restype = None
    lib.oracle_dequantize_grad_int8.argtypes = [p, p, i64, i32, p]
    lib.oracle_dequantize_grad_int8.restype = None
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"expected bf16 bit patterns as uint16, got {a.dtype}"
    return a


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float32, f"expected float32, got {a.dtype}"
    return a


class AdamW:
    """AdamW hyper-parameters; every one of them an fp32 value."""

    def __init__(self, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1):
        self.lr = float(np.float32(lr))
        self.beta1 = float(np.float32(beta1))
        self.beta2 = float(np.float32(beta2))
        self.eps = float(np.float32(eps))
        self.weight_decay = float(np.float32(weight_decay))

    def args(self):
        return (self.lr, self.beta1, self.beta2, self.eps, self.weight_decay)


# --------------------------------------------------------------------------
# wrappers
# --------------------------------------------------------------------------

def bf16_to_f32(h) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def cast_bf16(x) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    x = _f32(x)
    y = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_cast_bf16(_ptr(x), _ptr(y), x.size)
    return y


def layout(numels, n_dp: int, align: int = 8, bucket: int = 500_000_000):
    """Returns dict(n, shard, padded, bucket, n_buckets, offsets) or raises ValueError."""
    numel = np.ascontiguousarray(np.asarray(numels, dtype=np.int64).reshape(-1))
    offsets = np.zeros(max(numel.size, 1), dtype=np.int64)
    out = np.zeros(5, dtype=np.int64)
    rc = _load().oracle_layout(_ptr(numel) if numel.size else None, numel.size, n_dp, align,
                               bucket, _ptr(offsets), _ptr(out))
    if rc != 0:
        raise ValueError(f"no layout for n_dp={n_dp} align={align} bucket={bucket} (rc={rc})")
    n, s, p, bq, nb = (int(x) for x in out)
    return dict(n=n, shard=s, padded=p, bucket=bq, n_buckets=nb,
                offsets=offsets[: numel.size].copy())


def reduce_mean(src, divisor: float) -> np.ndarray:
    """Mean over rows (ranks) of a 2-D array: bf16 (uint16) or fp32 rows."""
    src = np.ascontiguousarray(src)
    assert src.ndim == 2
    n_src, n = src.shape
    g = np.empty(n, dtype=np.float32)
    if src.dtype == np.uint16:
        _load().oracle_reduce_mean_bf16(_ptr(src), n_src, n, n, float(np.float32(divisor)), _ptr(g))
    else:
        src = _f32(src)
        _load().oracle_reduce_mean_f32(_ptr(src), n_src, n, n, float(np.float32(divisor)), _ptr(g))
    return g


def bias_corrections(hp: AdamW, t: int):
    b1 = ctypes.c_float()
    b2 = ctypes.c_float()
    _load().oracle_bias_corrections(hp.beta1, hp.beta2, t, ctypes.byref(b1), ctypes.byref(b2))
    return np.float32(b1.value), np.float32(b2.value)


def adamw(w, m, v, g, hp: AdamW, t: int):
    """Returns new (w, m, v); the inputs are not modified."""
    w = _f32(w).copy()
    m = _f32(m).copy()
    v = _f32(v).copy()
    g = _f32(g)
    assert w.shape == m.shape == v.shape == g.shape
    _load().oracle_adamw(_ptr(w), _ptr(m), _ptr(v), _ptr(g), w.size, *hp.args(), t)
    return w, m, v


def zero_step(grads, w_shards, m_shards, v_shards, hp: AdamW, t: int, n_copies: int = 1):
    """ZeRO-1/2 step over n_dp simulated ranks.

    grads: (n_dp, P) uint16 bf16; w/m/v_shards: (n_dp, S) fp32.
    Returns (full_w (n_copies, P) uint16, w, m, v) -- new arrays, inputs untouched.
    """
    grads = _u16(grads)
    n_dp, p = grads.shape
    w = _f32(w_shards).copy()
    m = _f32(m_shards).copy()
    v = _f32(v_shards).copy()
    assert w.shape == (n_dp, p // n_dp) and p % n_dp == 0
    s = p // n_dp
    full = np.empty((n_copies, p), dtype=np.uint16)
    rc = _load().oracle_zero_step(_ptr(grads), n_dp, s, _ptr(w), _ptr(m), _ptr(v), _ptr(full),
                                  n_copies, *hp.args(), t)
    assert rc == 0, rc
    return full, w, m, v


def dp_step(grads, w_full, m_full, v_full, hp: AdamW, t: int):
    """Plain data parallelism: every rank holds (n_dp, P) full copies."""
    grads = _u16(grads)
    n_dp, p = grads.shape
    w = _f32(w_full).copy()
    m = _f32(m_full).copy()
    v = _f32(v_full).copy()
    assert w.shape == (n_dp, p)
    full = np.empty((n_dp, p), dtype=np.uint16)
    rc = _load().oracle_dp_step(_ptr(grads), n_dp, p, _ptr(w), _ptr(m), _ptr(v), _ptr(full),
                                *hp.args(), t)
    assert rc == 0, rc
    return full, w, m, v


def accumulate_local(acc, g, first: bool) -> np.ndarray:
    g = _u16(g)
    acc = np.zeros(g.shape, np.float32) if acc is None else _f32(acc).copy()
    _load().oracle_accumulate_local(_ptr(acc), _ptr(g), g.size, int(bool(first)))
    return acc


def accumulate_reduce(acc, src, first: bool) -> np.ndarray:
    src = _u16(src)
    n_src, n = src.shape
    acc = np.zeros(n, np.float32) if acc is None else _f32(acc).copy()
    _load().oracle_accumulate_reduce(_ptr(acc), _ptr(src), n_src, n, n, int(bool(first)))
    return acc


def all_gather(shards) -> np.ndarray:
    shards = _u16(shards)
    n_dp, s = shards.shape
    full = np.empty(n_dp * s, dtype=np.uint16)
    _load().oracle_all_gather_bf16(_ptr(shards), n_dp, s, _ptr(full))
    return full


def grad_norm_sq(src, divisor) -> float:
    """Squared L2 norm (fp64) of the mean over rows of a 2-D array."""
    src = np.ascontiguousarray(src)
    n_src, n = src.shape
    d = float(np.float32(divisor))
    if src.dtype == np.uint16:
        return _load().oracle_grad_norm_sq_bf16(_ptr(src), n_src, n, n, d)
    src = _f32(src)
    return _load().oracle_grad_norm_sq_f32(_ptr(src), n_src, n, n, d)


def clip_coef(norm_sq: float, max_norm: float) -> np.float32:
    return np.float32(_load().oracle_clip_coef(float(norm_sq), float(np.float32(max_norm))))


def scale(g, coef) -> np.ndarray:
    g = _f32(g).copy()
    _load().oracle_scale(_ptr(g), g.size, float(np.float32(coef)))
    return g


def rs_adamw_reference(src, divisor, w, m, v, hp: AdamW, t: int, clip=None):
    """Mean of source rows, (optionally) the clip scale, then AdamW, then cast:
    the per-element definition of one fused update call.  clip = (norm_sq,
    max_norm) with norm_sq the squared norm of the whole step's mean gradient.
    Returns (out_bf16, w, m, v)."""
    g = reduce_mean(src, divisor)
    if clip is not None:
        g = scale(g, clip_coef(*clip))
    w2, m2, v2 = adamw(w, m, v, g, hp, t)
    return cast_bf16(w2), w2, m2, v2


def quantize_int8(w_bf16, block: int = 256):
    """One shard's bf16 weights -> (int8 q, fp32 per-block scales)."""
    w = _u16(w_bf16).reshape(-1)
    nb = -(-w.size // block)
    q = np.empty(w.size, dtype=np.int8)
    scales = np.empty(max(nb, 1), dtype=np.float32)
    _load().oracle_quantize_int8(_ptr(w), w.size, block, _ptr(q), _ptr(scales))
    return q, scales[:nb]


def dequantize_int8(q, scales, block: int = 256):
    q = np.ascontiguousarray(q, dtype=np.int8).reshape(-1)
    scales = _f32(scales)
    out = np.empty(q.size, dtype=np.uint16)
    _load().oracle_dequantize_int8(_ptr(q), _ptr(scales), q.size, block, _ptr(out))
    return out


# ---------------------------------------------------------------------------
# 8-bit quantized gradient reduce-scatter (ZeRO++): "ZeRO Optimizer, in depth",
# "Offload and ZeRO++" (zero_quantized_gradients); "ZeRO and FSDP", "Fewer
# bytes on the wire".  Each rank's gradient slice for owner o is quantized in
# the weight format; the owner dequantizes to fp32 and takes the fp32 mean.
# ---------------------------------------------------------------------------

def quantize_grad_int8(g_rows, n_dp: int, block: int = 256):
    """Rows of bf16 gradients (n_src, P = n_dp*S), every row quantized slice by
    slice (slice o = [o*S, (o+1)*S)) -> q (n_src, P) int8 and scales
    (n_src, n_dp*nb) fp32 with nb = ceil(S / block), slice o's at [o*nb]."""
    g = _u16(g_rows)
    assert g.ndim == 2 and g.shape[1] % n_dp == 0
    n_src, P = g.shape
    S = P // n_dp
    nb = -(-S // block)
    q = np.empty((n_src, P), dtype=np.int8)
    scales = np.empty((n_src, n_dp * nb), dtype=np.float32)
    for r in range(n_src):
        for o in range(n_dp):
            q[r, o * S:(o + 1) * S], scales[r, o * nb:(o + 1) * nb] = \
                quantize_int8(g[r, o * S:(o + 1) * S], block)
    return q, scales


def dequantize_grad_int8(q_rows, scale_rows, n_dp: int, block: int = 256) -> np.ndarray:
    """The owners' fp32 view of quantized gradient rows: (n_src, P) float32,
    element k of slice o = code * (slice o's scale of block k // block)."""
    q = np.ascontiguousarray(q_rows, dtype=np.int8)
    sc = _f32(scale_rows)
    n_src, P = q.shape
    S = P // n_dp
    nb = -(-S // block)
    assert sc.shape == (n_src, n_dp * nb)
    out = np.empty((n_src, P), dtype=np.float32)
    for r in range(n_src):
        for o in range(n_dp):
            qs = np.ascontiguousarray(q[r, o * S:(o + 1) * S])
            ss = np.ascontiguousarray(sc[r, o * nb:(o + 1) * nb])
            part = np.empty(S, dtype=np.float32)
            _load().oracle_dequantize_grad_int8(_ptr(qs), _ptr(ss), S, block, _ptr(part))
            out[r, o * S:(o + 1) * S] = part
    return out


def qgrad_rs_adamw_reference(q_rows, scale_rows, n_dp: int, block: int, divisor, w, m, v,
                             hp: AdamW, t: int):
    """One step over the whole padded vector from 8-bit gradients: dequantize,
    fp32 mean over ranks, AdamW, bf16 cast.  Returns (out_bf16, w, m, v)."""
    g = reduce_mean(dequantize_grad_int8(q_rows, scale_rows, n_dp, block), divisor)
    w2, m2, v2 = adamw(w, m, v, g, hp, t)
    return cast_bf16(w2), w2, m2, v2


def accumulate_reduce_int8(acc, q_rows, scale_rows, n_dp: int, block: int, first: bool) -> np.ndarray:
    """The owner's fp32 accumulation of 8-bit gradients over the whole padded
    vector: x = +0 + sum over ranks of the dequantized values (ascending), then
    acc = x (first) or acc + x (one fp32 addition)."""
    x = reduce_mean(dequantize_grad_int8(q_rows, scale_rows, n_dp, block), 1.0)   # sum / 1 is exact
    if first:
        return x
    return (_f32(acc) + x).astype(np.float32)
