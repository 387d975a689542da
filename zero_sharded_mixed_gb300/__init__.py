"""ZeRO stage-1/2/3 sharded mixed-precision step for GB300 (sm_103a).

The compute lives in ``libzero_gb300.so`` (hand-written CUDA kernels behind a
C ABI, declared in ``include/zero_gb300.h``); ``binding`` is a thin ctypes layer
with the same names.  The library is loaded on first use of a binding name, so
importing ``zero_sharded_mixed_gb300.inputs`` alone does not need a GPU or a
built library.  There is no CPU fallback: if the library is missing, every
binding call raises.
"""
from __future__ import annotations

_BINDING_NAMES = {
    "ZeroError", "ZeroLayout", "ZeroAdamW", "lib_path", "load",
    "zero_layout", "zero_reduce_scatter_adamw", "zero_gather_layer", "zero_accumulate", "zero_cast_bf16",
    "zero_reduce_scatter_adamw_clip", "zero_accumulate_adamw", "zero_grad_norm_workspace",
    "zero_grad_norm_sq", "zero_grad_norm_sq_static", "zero_quantize_int8", "zero_gather_layer_int8",
    "zero_reduce_scatter_adamw_int8", "zero_accumulate_int8", "zero_reduce_scatter_adamw_q8",
    "zero_reduce_scatter_adamw_int8_q8", "zero_schedule_fill", "zero_schedule_advance",
    "zero_status_check", "zero_strerror", "zero_memory_bytes", "zero_comm_bytes",
    "zero_bucket_range", "zero_shard_range", "zero_selftest_bounded_wait", "zero_lr_warmup_decay",
    "ZERO_OK", "ZERO_EINVAL", "ZERO_EALIGN", "ZERO_ERANGE", "ZERO_ECUDA", "ZERO_ETIMEOUT",
    "ZERO_EIO", "ZERO_ECORRUPT",
    "ZERO_BF16", "ZERO_F32", "ZERO_OUT_FULL", "ZERO_OUT_SHARD",
    "ZERO_ACC_LOCAL", "ZERO_ACC_REDUCE", "ZERO_MAX_SRC",
}


_ENGINE_NAMES = {"ZeroEngine", "Zero3Engine"}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    if name in _ENGINE_NAMES:
        from . import engine
        return getattr(engine, name)
    if name == "ZeroConfig":
        from .config import ZeroConfig
        return ZeroConfig
    raise AttributeError(name)
