"""The subset of a DeepSpeed configuration that the ZeRO step reads.

"DeepSpeed ZeRO", "The configuration file" and "ZeRO Optimizer, in depth",
"Running it with DeepSpeed": a JSON configuration names the ZeRO stage, the
reduce bucket size, the number of gradient-accumulation steps, the clipping
threshold, the optimizer (AdamW with lr, betas, eps, weight_decay) and the
precision (bf16), and a "WarmupDecayLR" learning-rate scheduler; "Offload and
ZeRO++" adds zero_quantized_weights and zero_quantized_gradients.  ``ZeroConfig.from_dict`` reads those keys, refuses
what the library does not do (fp16 loss scaling, offload, another optimizer),
and lists the keys it did not use instead of failing on them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

_USED_TOP = {"zero_optimization", "optimizer", "gradient_accumulation_steps", "gradient_clipping",
             "bf16", "fp16", "scheduler"}
_USED_ZERO = {"stage", "reduce_bucket_size", "zero_quantized_weights", "zero_quantized_gradients",
              "offload_optimizer", "offload_param", "overlap_comm",
              "stage3_gather_16bit_weights_on_model_save"}


@dataclass
class ZeroConfig:
    stage: int = 2
    reduce_bucket_size: int = 500_000_000
    gradient_accumulation_steps: int = 1
    gradient_clipping: float = 0.0            # 0: no clipping
    lr: float = 1e-4
    betas: tuple = (0.9, 0.999)
    eps: float = 1e-8
    weight_decay: float = 0.0
    zero_quantized_weights: bool = False      # stage 3: 8-bit weight gathers
    zero_quantized_gradients: bool = False    # 8-bit gradient reduce-scatter
    overlap_comm: bool = False                # stage 3: gathers one unit ahead on a side stream
    stage3_gather_16bit_weights_on_model_save: bool = False   # stage 3: save_16bit_model allowed
    quant_block: int = 256
    # WarmupDecayLR: {"min_lr", "max_lr", "warmup_steps", "total_steps"}, or None for a constant lr
    scheduler: dict | None = None
    ignored: list = field(default_factory=list)

    def __post_init__(self):
        if self.stage not in (1, 2, 3):
            raise ValueError(f"zero_optimization.stage must be 1, 2 or 3, got {self.stage!r}")
        if self.reduce_bucket_size < 1:
            raise ValueError("reduce_bucket_size must be positive")
        if self.gradient_accumulation_steps < 1:
            raise ValueError("gradient_accumulation_steps must be at least 1")
        if self.gradient_clipping < 0:
            raise ValueError("gradient_clipping must be 0 (off) or positive")
        if self.zero_quantized_weights and self.stage != 3:
            raise ValueError("zero_quantized_weights applies to stage 3 (the weight all-gather)")
        if not (0.0 <= self.betas[0] < 1.0 and 0.0 <= self.betas[1] < 1.0):
            raise ValueError(f"betas must lie in [0, 1), got {self.betas!r}")
        if self.scheduler is not None:
            sc = self.scheduler
            if not (0 <= sc["warmup_steps"] < sc["total_steps"]):
                raise ValueError("the scheduler needs 0 <= warmup_num_steps < total_num_steps")
            if not (sc["min_lr"] >= 0.0 and sc["max_lr"] >= 0.0):
                raise ValueError("the scheduler's learning rates must be non-negative")

    def lr_at(self, t: int) -> float:
        """The learning rate of optimizer step t (t >= 1): the optimizer's lr, or
        the scheduler's value at that step (computed by the library)."""
        if self.scheduler is None:
            return self.lr
        from . import binding
        sc = self.scheduler
        return binding.zero_lr_warmup_decay(t, sc["min_lr"], sc["max_lr"], sc["warmup_steps"],
                                            sc["total_steps"])

    @classmethod
    def from_dict(cls, cfg: dict) -> "ZeroConfig":
        zo = dict(cfg.get("zero_optimization", {}))
        for key in ("offload_optimizer", "offload_param"):
            dev = (zo.get(key) or {}).get("device", "none")
            if dev not in ("none", None):
                raise ValueError(f"zero_optimization.{key} to {dev!r}: offload is not supported by this library")
        if (cfg.get("fp16") or {}).get("enabled", False):
            raise ValueError("fp16 with loss scaling is not supported by this library: use bf16")
        if not (cfg.get("bf16") or {"enabled": True}).get("enabled", True):
            raise ValueError("this library keeps weights and gradients in bf16: bf16.enabled must be true")
        opt = cfg.get("optimizer") or {"type": "AdamW", "params": {}}
        if str(opt.get("type", "AdamW")).lower() != "adamw":
            raise ValueError(f"optimizer {opt.get('type')!r}: this library implements AdamW")
        p = opt.get("params", {})
        scheduler = None
        if cfg.get("scheduler") is not None:
            sch = cfg["scheduler"]
            if sch.get("type") != "WarmupDecayLR":
                raise ValueError(f"scheduler {sch.get('type')!r}: this library implements WarmupDecayLR")
            sp = sch.get("params", {})
            if sp.get("warmup_type", "linear") != "linear":
                raise ValueError("WarmupDecayLR is implemented with a linear warmup")
            missing = [k for k in ("warmup_num_steps", "total_num_steps") if k not in sp]
            if missing:
                raise ValueError(f"WarmupDecayLR needs {', '.join(missing)}")
            scheduler = {"min_lr": float(sp.get("warmup_min_lr", 0.0)),
                         "max_lr": float(sp.get("warmup_max_lr", p.get("lr", 1e-4))),
                         "warmup_steps": int(sp["warmup_num_steps"]),
                         "total_steps": int(sp["total_num_steps"])}
        ignored = sorted([k for k in cfg if k not in _USED_TOP] +
                         [f"zero_optimization.{k}" for k in zo if k not in _USED_ZERO])
        return cls(
            stage=int(zo.get("stage", 2)),
            reduce_bucket_size=int(float(zo.get("reduce_bucket_size", 5e8))),
            gradient_accumulation_steps=int(cfg.get("gradient_accumulation_steps", 1)),
            gradient_clipping=float(cfg.get("gradient_clipping", 0.0)),
            lr=float(p.get("lr", 1e-4)),
            betas=tuple(float(b) for b in p.get("betas", (0.9, 0.999))),
            eps=float(p.get("eps", 1e-8)),
            weight_decay=float(p.get("weight_decay", 0.0)),
            zero_quantized_weights=bool(zo.get("zero_quantized_weights", False)),
            zero_quantized_gradients=bool(zo.get("zero_quantized_gradients", False)),
            overlap_comm=bool(zo.get("overlap_comm", False)),
            stage3_gather_16bit_weights_on_model_save=bool(
                zo.get("stage3_gather_16bit_weights_on_model_save", False)),
            scheduler=scheduler,
            ignored=ignored,
        )
