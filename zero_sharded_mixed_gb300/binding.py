"""Thin ctypes binding for libzero_gb300.so (names as in include/zero_gb300.h).

Argument marshalling only: torch tensors are checked (device, dtype,
contiguity, extent) and turned into pointers; every step of the computation
runs in the library's CUDA kernels.  There is no CPU fallback: if the library
is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libzero_gb300.so")

ZERO_OK, ZERO_EINVAL, ZERO_EALIGN, ZERO_ERANGE, ZERO_ECUDA, ZERO_ETIMEOUT = 0, -1, -2, -3, -4, -5
ZERO_EIO, ZERO_ECORRUPT = -6, -7
ZERO_BF16, ZERO_F32 = 0, 1
ZERO_OUT_FULL, ZERO_OUT_SHARD = 0, 1
ZERO_ACC_LOCAL, ZERO_ACC_REDUCE = 0, 1
ZERO_MAX_SRC = 64


class ZeroError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if code == ZERO_ECUDA:
            detail = f" [{load().zero_last_cuda_error().decode()}]"
        super().__init__(f"{where}: {zero_strerror(code)} ({code}){detail}")


class ZeroLayout(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("padded_n", ctypes.c_int64), ("shard", ctypes.c_int64),
                ("align", ctypes.c_int64), ("bucket", ctypes.c_int64), ("n_buckets", ctypes.c_int64),
                ("n_dp", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}

    def __repr__(self):
        return f"ZeroLayout({self.as_dict()})"


class ZeroCkptHeader(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("padded_n", ctypes.c_int64), ("shard", ctypes.c_int64),
                ("align", ctypes.c_int64), ("step", ctypes.c_int64), ("n_dp", ctypes.c_int32),
                ("rank", ctypes.c_int32), ("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("reserved", ctypes.c_int32)]


class ZeroAdamW(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("reserved", ctypes.c_int32), ("step", ctypes.c_int64),
                ("sched", ctypes.c_void_p)]

    @classmethod
    def make(cls, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, step=1, sched=None):
        """sched: None, or a CUDA float32 tensor of 3 elements {lr, bc1, bc2}
        that the kernels read in place of lr and step.  The block keeps a
        reference to it, so the memory outlives every call made with the block."""
        ptr = None
        if sched is not None:
            ptr = _tensor(sched, "sched", torch.float32, 3)
        hp = cls(lr, beta1, beta2, eps, weight_decay, 0, step, ptr)
        hp._sched_tensor = sched
        return hp


_lock = threading.Lock()
_lib = None


def load():
    """Load the library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(lib_path):
            raise ImportError(
                f"{lib_path} is missing: build it with `python -m zero_sharded_mixed_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(lib_path)
        i32, i64, f32, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
        P = ctypes.POINTER
        lib.zero_layout.argtypes = [P(i64), i32, i32, i64, i64, P(i64), P(ZeroLayout)]
        lib.zero_bucket_range.argtypes = [P(ZeroLayout), i64, P(i64), P(i64)]
        lib.zero_shard_range.argtypes = [P(ZeroLayout), i32, P(i64), P(i64), P(i64)]
        lib.zero_reduce_scatter_adamw.argtypes = [
            P(ZeroLayout), P(p), i32, i32, i64, f32, i32, i32, i64, i64,
            p, p, p, p, i32, P(ZeroAdamW), p]
        lib.zero_reduce_scatter_adamw_clip.argtypes = [
            P(ZeroLayout), P(p), i32, i32, i64, f32, i32, i32, i64, i64,
            p, p, p, p, i32, P(ZeroAdamW), p, f32, p]
        lib.zero_accumulate_adamw.argtypes = [
            P(ZeroLayout), i32, P(p), i32, i64, P(p), i32, i64, f32, i32, i32, i64, i64,
            p, p, p, p, i32, P(ZeroAdamW), p]
        lib.zero_grad_norm_workspace.argtypes = [P(i64)]
        lib.zero_grad_norm_sq.argtypes = [P(ZeroLayout), P(p), i32, i32, i64, f32, i64, i64,
                                          p, i64, p, i32, p]
        lib.zero_grad_norm_sq_static.argtypes = [P(ZeroLayout), P(p), i32, i32, i64, f32, i64,
                                                 i64, p, i32, p]
        lib.zero_gather_layer.argtypes = [P(ZeroLayout), P(p), p, p]
        lib.zero_cast_bf16.argtypes = [p, p, i64, p]
        lib.zero_quantize_int8.argtypes = [P(ZeroLayout), p, p, p, i32, p]
        lib.zero_ckpt_write_shard.argtypes = [ctypes.c_char_p, P(ZeroCkptHeader), p, p, p, p]
        lib.zero_ckpt_read_header.argtypes = [ctypes.c_char_p, P(ZeroCkptHeader), P(i32)]
        lib.zero_ckpt_read_shard.argtypes = [ctypes.c_char_p, P(ZeroCkptHeader), p, p, p, p, i64]
        lib.zero_selftest_bounded_wait.argtypes = [i64, p]
        lib.zero_schedule_fill.argtypes = [P(ZeroAdamW), i64, i64, p, p]
        lib.zero_schedule_advance.argtypes = [p, i64, p, p, p]
        lib.zero_crc32.argtypes = [p, i64]
        lib.zero_ckpt_payload_crc.argtypes = [ctypes.c_char_p, P(ctypes.c_uint32)]
        lib.zero_crc32.restype = ctypes.c_uint32
        lib.zero_gather_layer_int8.argtypes = [P(ZeroLayout), P(p), P(p), i32, p, p]
        lib.zero_reduce_scatter_adamw_q8.argtypes = [
            P(ZeroLayout), P(p), i32, i32, i64, f32, i32, i32, i64, i64,
            p, p, p, p, p, i32, P(ZeroAdamW), p]
        lib.zero_reduce_scatter_adamw_int8_q8.argtypes = [
            P(ZeroLayout), P(p), P(p), i32, i32, f32, i32, i32, i64, i64,
            p, p, p, p, p, i32, P(ZeroAdamW), p]
        lib.zero_reduce_scatter_adamw_int8.argtypes = [
            P(ZeroLayout), P(p), P(p), i32, i32, f32, i32, i32, i64, i64,
            p, p, p, p, i32, P(ZeroAdamW), p]
        lib.zero_accumulate_int8.argtypes = [P(ZeroLayout), P(p), P(p), i32, i32, p, i64, i64, i64,
                                             i32, p]
        lib.zero_accumulate.argtypes = [P(ZeroLayout), i32, P(p), i32, i32, i64, p, i64, i64, i64,
                                        i32, p]
        lib.zero_status_check.argtypes = [p]
        lib.zero_strerror.argtypes = [ctypes.c_int]
        lib.zero_strerror.restype = ctypes.c_char_p
        lib.zero_last_cuda_error.argtypes = []
        lib.zero_last_cuda_error.restype = ctypes.c_char_p
        lib.zero_memory_bytes.argtypes = [ctypes.c_double, i32, i32, ctypes.c_double,
                                          P(ctypes.c_double)]
        lib.zero_comm_bytes.argtypes = [ctypes.c_double, i32, i32, ctypes.c_double,
                                        ctypes.c_double, P(ctypes.c_double)]
        lib.zero_lr_warmup_decay.argtypes = [i64, ctypes.c_double, ctypes.c_double, i64, i64, P(f32)]
        for name in ("zero_layout", "zero_bucket_range", "zero_shard_range",
                     "zero_reduce_scatter_adamw", "zero_reduce_scatter_adamw_clip",
                     "zero_accumulate_adamw", "zero_grad_norm_workspace", "zero_grad_norm_sq",
                     "zero_grad_norm_sq_static", "zero_quantize_int8", "zero_gather_layer_int8",
                     "zero_ckpt_write_shard", "zero_ckpt_read_header", "zero_ckpt_read_shard",
                     "zero_ckpt_payload_crc",
                     "zero_selftest_bounded_wait", "zero_reduce_scatter_adamw_int8",
                     "zero_reduce_scatter_adamw_q8", "zero_reduce_scatter_adamw_int8_q8",
                     "zero_schedule_fill", "zero_schedule_advance",
                     "zero_accumulate_int8", "zero_gather_layer", "zero_accumulate",
                     "zero_status_check", "zero_memory_bytes", "zero_comm_bytes",
                     "zero_lr_warmup_decay"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def zero_strerror(code: int) -> str:
    return load().zero_strerror(int(code)).decode()


def _check(rc: int, where: str):
    if rc != ZERO_OK:
        raise ZeroError(rc, where)


# --------------------------------------------------------------------------
# host-only calls
# --------------------------------------------------------------------------

def zero_layout(numels: Sequence[int], n_dp: int, align: int = 8,
                bucket_elems: int = 500_000_000, with_offsets: bool = False):
    arr = (ctypes.c_int64 * max(1, len(numels)))(*[int(x) for x in numels])
    offs = (ctypes.c_int64 * max(1, len(numels)))()
    L = ZeroLayout()
    _check(load().zero_layout(arr, len(numels), int(n_dp), int(align), int(bucket_elems), offs,
                              ctypes.byref(L)), "zero_layout")
    if with_offsets:
        return L, [offs[i] for i in range(len(numels))]
    return L


def zero_bucket_range(L: ZeroLayout, b: int):
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    _check(load().zero_bucket_range(ctypes.byref(L), int(b), ctypes.byref(lo), ctypes.byref(hi)),
           "zero_bucket_range")
    return lo.value, hi.value


def zero_shard_range(L: ZeroLayout, rank: int):
    lo, hi, valid = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(load().zero_shard_range(ctypes.byref(L), int(rank), ctypes.byref(lo), ctypes.byref(hi),
                                   ctypes.byref(valid)), "zero_shard_range")
    return lo.value, hi.value, valid.value


def zero_lr_warmup_decay(t: int, min_lr: float, max_lr: float, warmup_steps: int,
                         total_steps: int) -> float:
    """The learning rate of optimizer step t (>= 1) under WarmupDecayLR."""
    out = ctypes.c_float()
    _check(load().zero_lr_warmup_decay(int(t), float(min_lr), float(max_lr), int(warmup_steps),
                                       int(total_steps), ctypes.byref(out)), "zero_lr_warmup_decay")
    return out.value


def zero_memory_bytes(n, n_dp, stage, k_bytes=12.0) -> float:
    out = ctypes.c_double()
    _check(load().zero_memory_bytes(float(n), int(n_dp), int(stage), float(k_bytes),
                                    ctypes.byref(out)), "zero_memory_bytes")
    return out.value


def zero_comm_bytes(n, n_dp, stage, param_bytes=2.0, grad_bytes=2.0) -> float:
    out = ctypes.c_double()
    _check(load().zero_comm_bytes(float(n), int(n_dp), int(stage), float(param_bytes),
                                  float(grad_bytes), ctypes.byref(out)), "zero_comm_bytes")
    return out.value


# --------------------------------------------------------------------------
# device calls
# --------------------------------------------------------------------------

def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _tensor(t: torch.Tensor, name: str, dtype, min_numel: int, pinned_ok: bool = False) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if pinned_ok and t.device.type == "cpu":
        if not t.is_pinned():
            raise ValueError(f"{name} is host memory but not pinned; the kernels read only "
                             "device memory or pinned host memory")
    elif t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device}); there is no CPU path")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < min_numel:
        raise ValueError(f"{name} has {t.numel()} elements, the call reads or writes {min_numel}")
    return t.data_ptr()


_SRC_DT = {ZERO_BF16: torch.bfloat16, ZERO_F32: torch.float32}


def _src_array(srcs, dtype, min_numel, pinned_ok=False):
    if len(srcs) == 0:
        raise ValueError("need at least one source")
    ptrs = [_tensor(s, f"src[{i}]", dtype, min_numel, pinned_ok) for i, s in enumerate(srcs)]
    return (ctypes.c_void_p * len(ptrs))(*ptrs), len(ptrs)


def zero_reduce_scatter_adamw(L: ZeroLayout, srcs, src_dtype: int, src_base: int, divisor: float,
                              rank_begin: int, rank_end: int, begin: int, end: int,
                              master: torch.Tensor, m: torch.Tensor, v: torch.Tensor,
                              out: torch.Tensor, out_mode: int, hp: ZeroAdamW, stream=None):
    """Fused mean reduce-scatter + AdamW + bf16 cast + gather write over [begin, end).
    The sources may be pinned host tensors: the kernel then reads them over the
    host link."""
    if end <= begin:
        src_need = state_need = out_need = 0
    else:
        src_need = end - src_base
        state_need = end - rank_begin * L.shard
        out_need = end if out_mode == ZERO_OUT_FULL else state_need
    arr, n = _src_array(srcs, _SRC_DT.get(src_dtype, None), src_need, pinned_ok=True)
    rc = load().zero_reduce_scatter_adamw(
        ctypes.byref(L), arr, n, int(src_dtype), int(src_base), float(divisor),
        int(rank_begin), int(rank_end), int(begin), int(end),
        _tensor(master, "master", torch.float32, state_need),
        _tensor(m, "m", torch.float32, state_need),
        _tensor(v, "v", torch.float32, state_need),
        _tensor(out, "out", torch.bfloat16, out_need),
        int(out_mode), ctypes.byref(hp), _stream_ptr(stream))
    _check(rc, "zero_reduce_scatter_adamw")


def zero_reduce_scatter_adamw_clip(L: ZeroLayout, srcs, src_dtype: int, src_base: int,
                                   divisor: float, rank_begin: int, rank_end: int, begin: int,
                                   end: int, master: torch.Tensor, m: torch.Tensor,
                                   v: torch.Tensor, out: torch.Tensor, out_mode: int,
                                   hp: ZeroAdamW, norm_sq: torch.Tensor, max_norm: float,
                                   stream=None):
    """zero_reduce_scatter_adamw with the mean gradient scaled by
    min(1, max_norm / (sqrt(norm_sq) + 1e-6)); norm_sq is a 1-element fp64 CUDA tensor."""
    if end <= begin:
        src_need = state_need = out_need = 0
    else:
        src_need = end - src_base
        state_need = end - rank_begin * L.shard
        out_need = end if out_mode == ZERO_OUT_FULL else state_need
    arr, n = _src_array(srcs, _SRC_DT.get(src_dtype, None), src_need, pinned_ok=True)
    rc = load().zero_reduce_scatter_adamw_clip(
        ctypes.byref(L), arr, n, int(src_dtype), int(src_base), float(divisor),
        int(rank_begin), int(rank_end), int(begin), int(end),
        _tensor(master, "master", torch.float32, state_need),
        _tensor(m, "m", torch.float32, state_need),
        _tensor(v, "v", torch.float32, state_need),
        _tensor(out, "out", torch.bfloat16, out_need),
        int(out_mode), ctypes.byref(hp), _tensor(norm_sq, "norm_sq", torch.float64, 1),
        float(max_norm), _stream_ptr(stream))
    _check(rc, "zero_reduce_scatter_adamw_clip")


def zero_reduce_scatter_adamw_q8(L: ZeroLayout, srcs, src_dtype: int, src_base: int,
                                 divisor: float, rank_begin: int, rank_end: int, begin: int,
                                 end: int, master: torch.Tensor, m: torch.Tensor, v: torch.Tensor,
                                 q_out: torch.Tensor, scales_out: torch.Tensor, block: int,
                                 hp: ZeroAdamW, stream=None):
    """The fused update with its result in the 8-bit block format (codes laid
    out like the state, one scale per 256 of them) instead of bf16."""
    if end <= begin:
        src_need = state_need = 0
    else:
        src_need = end - src_base
        state_need = end - rank_begin * L.shard
    arr, n = _src_array(srcs, _SRC_DT.get(src_dtype, None), src_need)
    rc = load().zero_reduce_scatter_adamw_q8(
        ctypes.byref(L), arr, n, int(src_dtype), int(src_base), float(divisor),
        int(rank_begin), int(rank_end), int(begin), int(end),
        _tensor(master, "master", torch.float32, state_need),
        _tensor(m, "m", torch.float32, state_need),
        _tensor(v, "v", torch.float32, state_need),
        _tensor(q_out, "q_out", torch.int8, state_need),
        _tensor(scales_out, "scales_out", torch.float32, -(-state_need // 256)),
        int(block), ctypes.byref(hp), _stream_ptr(stream))
    _check(rc, "zero_reduce_scatter_adamw_q8")


def zero_accumulate_adamw(L: ZeroLayout, mode: int, acc, acc_base: int, grads, grad_base: int,
                          divisor: float, rank_begin: int, rank_end: int, begin: int, end: int,
                          master: torch.Tensor, m: torch.Tensor, v: torch.Tensor,
                          out: torch.Tensor, out_mode: int, hp: ZeroAdamW, stream=None):
    """The last micro-batch of an accumulation window fused with the update
    (LOCAL: sum_r (acc[r] + grads[r]); REDUCE: acc[0] + sum_r grads[r])."""
    if end <= begin:
        acc_need = grad_need = state_need = out_need = 0
    else:
        acc_need, grad_need = end - acc_base, end - grad_base
        state_need = end - rank_begin * L.shard
        out_need = end if out_mode == ZERO_OUT_FULL else state_need
    if len(acc) == 0 or len(grads) == 0:
        raise ValueError("need accumulators and gradients")
    acc_p = [_tensor(a, f"acc[{i}]", torch.float32, acc_need) for i, a in enumerate(acc)]
    g_p = [_tensor(g, f"grads[{i}]", torch.bfloat16, grad_need) for i, g in enumerate(grads)]
    rc = load().zero_accumulate_adamw(
        ctypes.byref(L), int(mode), (ctypes.c_void_p * len(acc_p))(*acc_p), len(acc_p), int(acc_base),
        (ctypes.c_void_p * len(g_p))(*g_p), len(g_p), int(grad_base), float(divisor),
        int(rank_begin), int(rank_end), int(begin), int(end),
        _tensor(master, "master", torch.float32, state_need),
        _tensor(m, "m", torch.float32, state_need),
        _tensor(v, "v", torch.float32, state_need),
        _tensor(out, "out", torch.bfloat16, out_need),
        int(out_mode), ctypes.byref(hp), _stream_ptr(stream))
    _check(rc, "zero_accumulate_adamw")


def zero_grad_norm_workspace() -> int:
    """Bytes of device workspace zero_grad_norm_sq needs on the current device."""
    out = ctypes.c_int64()
    _check(load().zero_grad_norm_workspace(ctypes.byref(out)), "zero_grad_norm_workspace")
    return out.value


def zero_grad_norm_sq(L: ZeroLayout, srcs, src_dtype: int, src_base: int, divisor: float,
                      begin: int, end: int, workspace: torch.Tensor, norm_sq: torch.Tensor,
                      accumulate: bool, stream=None):
    """norm_sq (1-element fp64 CUDA tensor) (+)= sum over [begin, end) of the
    squared mean gradient; workspace: a CUDA tensor of zero_grad_norm_workspace() bytes."""
    src_need = max(0, end - src_base) if end > begin else 0
    arr, n = _src_array(srcs, _SRC_DT.get(src_dtype, None), src_need)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().zero_grad_norm_sq(ctypes.byref(L), arr, n, int(src_dtype), int(src_base),
                                  float(divisor), int(begin), int(end), workspace.data_ptr(),
                                  int(ws_bytes), _tensor(norm_sq, "norm_sq", torch.float64, 1),
                                  int(bool(accumulate)), _stream_ptr(stream))
    _check(rc, "zero_grad_norm_sq")


def zero_grad_norm_sq_static(L: ZeroLayout, srcs, src_dtype: int, src_base: int, divisor: float,
                             begin: int, end: int, norm_sq: torch.Tensor, accumulate: bool,
                             stream=None):
    """zero_grad_norm_sq with its partial sums in the library's own device array:
    no workspace, nothing allocated.  Calls that overlap on the GPU race."""
    src_need = max(0, end - src_base) if end > begin else 0
    arr, n = _src_array(srcs, _SRC_DT.get(src_dtype, None), src_need)
    rc = load().zero_grad_norm_sq_static(ctypes.byref(L), arr, n, int(src_dtype), int(src_base),
                                         float(divisor), int(begin), int(end),
                                         _tensor(norm_sq, "norm_sq", torch.float64, 1),
                                         int(bool(accumulate)), _stream_ptr(stream))
    _check(rc, "zero_grad_norm_sq_static")


def zero_gather_layer(unit: ZeroLayout, shards, full_out: torch.Tensor, stream=None):
    """Concatenate unit.n_dp bf16 shards (unit.shard elements each) into full_out."""
    if len(shards) != unit.n_dp:
        raise ValueError(f"need {unit.n_dp} shards, got {len(shards)}")
    ptrs = [_tensor(s, f"shards[{i}]", torch.bfloat16, unit.shard) for i, s in enumerate(shards)]
    arr = (ctypes.c_void_p * max(1, len(ptrs)))(*ptrs)
    rc = load().zero_gather_layer(ctypes.byref(unit), arr,
                                  _tensor(full_out, "full_out", torch.bfloat16, unit.padded_n),
                                  _stream_ptr(stream))
    _check(rc, "zero_gather_layer")


def zero_cast_bf16(src: torch.Tensor, dst: torch.Tensor, n: int = None, stream=None):
    """dst[:n] = bf16 of src[:n] (nearest, ties to even); n defaults to src.numel()."""
    n = src.numel() if n is None else int(n)
    rc = load().zero_cast_bf16(_tensor(src, "src", torch.float32, n), _tensor(dst, "dst", torch.bfloat16, n),
                               n, _stream_ptr(stream))
    _check(rc, "zero_cast_bf16")


def zero_accumulate(L: ZeroLayout, mode: int, srcs, src_dtype: int, src_base: int,
                    dst: torch.Tensor, dst_base: int, begin: int, end: int, first: bool,
                    stream=None):
    """dst[i - dst_base] (+)= src[0] (LOCAL) or sum_r src[r] (REDUCE) over [begin, end)."""
    src_need = max(0, end - src_base) if end > begin else 0
    dst_need = max(0, end - dst_base) if end > begin else 0
    arr, n = _src_array(srcs, _SRC_DT.get(src_dtype, None), src_need)
    rc = load().zero_accumulate(ctypes.byref(L), int(mode), arr, n, int(src_dtype), int(src_base),
                                _tensor(dst, "dst", torch.float32, dst_need), int(dst_base),
                                int(begin), int(end), int(bool(first)), _stream_ptr(stream))
    _check(rc, "zero_accumulate")


def zero_status_check(stream=None):
    _check(load().zero_status_check(_stream_ptr(stream)), "zero_status_check")


def zero_quantize_int8(unit: ZeroLayout, shards: torch.Tensor, q: torch.Tensor, scales: torch.Tensor,
                       block: int = 256, stream=None):
    """Quantize the unit's n_dp bf16 shards (back to back) to int8 + fp32 block scales."""
    nb = -(-unit.shard // block) if unit.shard else 0
    rc = load().zero_quantize_int8(
        ctypes.byref(unit), _tensor(shards, "shards", torch.bfloat16, unit.padded_n),
        _tensor(q, "q", torch.int8, unit.padded_n),
        _tensor(scales, "scales", torch.float32, nb * unit.n_dp), int(block), _stream_ptr(stream))
    _check(rc, "zero_quantize_int8")


def zero_gather_layer_int8(unit: ZeroLayout, q_shards, scale_shards, full_out: torch.Tensor,
                           block: int = 256, stream=None):
    """Rebuild the full bf16 unit from each rank's int8 shard and block scales."""
    if len(q_shards) != unit.n_dp or len(scale_shards) != unit.n_dp:
        raise ValueError(f"need {unit.n_dp} shards and scale arrays")
    nb = -(-unit.shard // block) if unit.shard else 0
    qp = [_tensor(x, f"q_shards[{i}]", torch.int8, unit.shard) for i, x in enumerate(q_shards)]
    sp = [_tensor(x, f"scale_shards[{i}]", torch.float32, nb) for i, x in enumerate(scale_shards)]
    rc = load().zero_gather_layer_int8(
        ctypes.byref(unit), (ctypes.c_void_p * max(1, len(qp)))(*qp),
        (ctypes.c_void_p * max(1, len(sp)))(*sp), int(block),
        _tensor(full_out, "full_out", torch.bfloat16, unit.padded_n), _stream_ptr(stream))
    _check(rc, "zero_gather_layer_int8")


def _qgrad_sources(L: ZeroLayout, q_src, scale_src, block: int, need: int):
    """Host arrays of the codes and scales of 8-bit gradient sources."""
    if len(q_src) == 0 or len(q_src) != len(scale_src):
        raise ValueError("need the same nonzero number of code and scale sources")
    nb = -(-L.shard // block) if L.shard else 0
    qp = [_tensor(x, f"q_src[{i}]", torch.int8, need) for i, x in enumerate(q_src)]
    sp = [_tensor(x, f"scale_src[{i}]", torch.float32, nb * L.n_dp if need else 0)
          for i, x in enumerate(scale_src)]
    n = len(qp)
    return (ctypes.c_void_p * n)(*qp), (ctypes.c_void_p * n)(*sp), n


def zero_reduce_scatter_adamw_int8(L: ZeroLayout, q_src, scale_src, block: int, divisor: float,
                                   rank_begin: int, rank_end: int, begin: int, end: int,
                                   master: torch.Tensor, m: torch.Tensor, v: torch.Tensor,
                                   out: torch.Tensor, out_mode: int, hp: ZeroAdamW, stream=None):
    """The fused update over [begin, end) from 8-bit gradients: each rank's
    codes (padded_n int8) and block scales (n_dp * ceil(S / block) fp32)."""
    if end <= begin:
        src_need = state_need = out_need = 0
    else:
        src_need = end
        state_need = end - rank_begin * L.shard
        out_need = end if out_mode == ZERO_OUT_FULL else state_need
    qa, sa, n = _qgrad_sources(L, q_src, scale_src, block, src_need)
    rc = load().zero_reduce_scatter_adamw_int8(
        ctypes.byref(L), qa, sa, n, int(block), float(divisor), int(rank_begin), int(rank_end),
        int(begin), int(end),
        _tensor(master, "master", torch.float32, state_need),
        _tensor(m, "m", torch.float32, state_need),
        _tensor(v, "v", torch.float32, state_need),
        _tensor(out, "out", torch.bfloat16, out_need),
        int(out_mode), ctypes.byref(hp), _stream_ptr(stream))
    _check(rc, "zero_reduce_scatter_adamw_int8")


def zero_reduce_scatter_adamw_int8_q8(L: ZeroLayout, q_src, scale_src, block: int, divisor: float,
                                      rank_begin: int, rank_end: int, begin: int, end: int,
                                      master: torch.Tensor, m: torch.Tensor, v: torch.Tensor,
                                      q_out: torch.Tensor, scales_out: torch.Tensor, out_block: int,
                                      hp: ZeroAdamW, stream=None):
    """The update from 8-bit gradients with its result in the 8-bit block format."""
    if end <= begin:
        src_need = state_need = 0
    else:
        src_need = end
        state_need = end - rank_begin * L.shard
    qa, sa, n = _qgrad_sources(L, q_src, scale_src, block, src_need)
    rc = load().zero_reduce_scatter_adamw_int8_q8(
        ctypes.byref(L), qa, sa, n, int(block), float(divisor), int(rank_begin), int(rank_end),
        int(begin), int(end),
        _tensor(master, "master", torch.float32, state_need),
        _tensor(m, "m", torch.float32, state_need),
        _tensor(v, "v", torch.float32, state_need),
        _tensor(q_out, "q_out", torch.int8, state_need),
        _tensor(scales_out, "scales_out", torch.float32, -(-state_need // 256)),
        int(out_block), ctypes.byref(hp), _stream_ptr(stream))
    _check(rc, "zero_reduce_scatter_adamw_int8_q8")


def zero_accumulate_int8(L: ZeroLayout, q_src, scale_src, block: int, dst: torch.Tensor,
                         dst_base: int, begin: int, end: int, first: bool, stream=None):
    """dst[i - dst_base] (+)= sum over ranks of the dequantized 8-bit gradients."""
    src_need = end if end > begin else 0
    dst_need = max(0, end - dst_base) if end > begin else 0
    qa, sa, n = _qgrad_sources(L, q_src, scale_src, block, src_need)
    rc = load().zero_accumulate_int8(ctypes.byref(L), qa, sa, n, int(block),
                                     _tensor(dst, "dst", torch.float32, dst_need), int(dst_base),
                                     int(begin), int(end), int(bool(first)), _stream_ptr(stream))
    _check(rc, "zero_accumulate_int8")


def zero_schedule_fill(hp: ZeroAdamW, first_step: int, n_steps: int, lrs=None) -> torch.Tensor:
    """Host table [n_steps, 3] of {lr, bc1, bc2} for steps first_step..; lrs: a
    sequence of n_steps learning rates, or None for hp.lr."""
    table = torch.empty((int(n_steps), 3), dtype=torch.float32)
    lr_arr = None
    if lrs is not None:
        lr_t = torch.tensor([float(x) for x in lrs], dtype=torch.float32)
        if lr_t.numel() != n_steps:
            raise ValueError(f"need {n_steps} learning rates, got {lr_t.numel()}")
        lr_arr = lr_t
    rc = load().zero_schedule_fill(ctypes.byref(hp), int(first_step), int(n_steps),
                                   lr_arr.data_ptr() if lr_arr is not None else None, table.data_ptr())
    _check(rc, "zero_schedule_fill")
    return table


def zero_schedule_advance(table: torch.Tensor, step_index: torch.Tensor, sched: torch.Tensor,
                          stream=None):
    """On the device: sched = table[step_index]; step_index += 1."""
    rc = load().zero_schedule_advance(_tensor(table, "table", torch.float32, 3),
                                      table.numel() // 3,
                                      _tensor(step_index, "step_index", torch.int64, 1),
                                      _tensor(sched, "sched", torch.float32, 3), _stream_ptr(stream))
    _check(rc, "zero_schedule_advance")


def zero_selftest_bounded_wait(limit_cycles: int, stream=None):
    """Run the bounded-wait self test (see zero_gb300.h); follow with zero_status_check."""
    _check(load().zero_selftest_bounded_wait(int(limit_cycles), _stream_ptr(stream)),
           "zero_selftest_bounded_wait")
