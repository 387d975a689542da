"""Model-state memory and communication volume per GPU for each ZeRO stage.

TEST INFRASTRUCTURE ONLY (part of the oracle).

Both follow "ZeRO and FSDP" (zerotofrontier.app):

* ``zero_memory`` -- section "Memory per GPU", the table of weights /
  gradients / optimizer bytes per stage, with 2-byte weights and gradients and
  K bytes of optimizer state per parameter; exercise "ZeRO memory per GPU"
  asks for a ValueError on any stage other than 0..3.
* ``zero_comm_bytes`` -- section "Communication volume" and exercise
  "Communication per step for each stage": ring collectives, a reduce-scatter
  or all-gather of an N-element vector sends (n_dp-1)/n_dp * N elements per
  GPU and an all-reduce twice that; stage 0 all-reduces gradients, stages 1
  and 2 reduce-scatter gradients and all-gather weights, stage 3 all-gathers
  weights twice and reduce-scatters gradients.

``warmup_decay_lr`` follows "DeepSpeed ZeRO", "The configuration file": the
example configuration's "WarmupDecayLR" scheduler with warmup_min_lr,
warmup_max_lr, warmup_num_steps and total_num_steps.  The page gives no
shape; the reading is linear warmup from the minimum to the maximum over the
warmup steps, then linear decay to 0 at total_num_steps, the first optimizer
step taking the value at 0 schedule steps.
"""
from __future__ import annotations

import numpy as np


def zero_memory(N, n_dp, stage, K=12):
    """Bytes of model states per GPU (weights + gradients + optimizer state)."""
    if stage not in (0, 1, 2, 3):
        raise ValueError(f"ZeRO stage must be 0, 1, 2 or 3, got {stage!r}")
    weights = 2 * N
    grads = 2 * N
    optimizer = K * N
    if stage >= 1:
        optimizer = optimizer / n_dp      # stage 1 shards the optimizer state
    if stage >= 2:
        grads = grads / n_dp              # stage 2 also shards the gradients
    if stage >= 3:
        weights = weights / n_dp          # stage 3 also shards the weights
    return weights + grads + optimizer


def zero_comm_bytes(N, n_dp, stage, param_bytes=2, grad_bytes=2):
    """Bytes each GPU sends per optimizer step under ring collectives."""
    if stage not in (0, 1, 2, 3):
        raise ValueError(f"ZeRO stage must be 0, 1, 2 or 3, got {stage!r}")
    one_pass = (n_dp - 1) / n_dp * N      # elements sent by one reduce-scatter or all-gather
    if stage == 0:
        return 2 * one_pass * grad_bytes                       # all-reduce of gradients
    if stage in (1, 2):
        return one_pass * grad_bytes + one_pass * param_bytes  # RS(grads) + AG(weights)
    return one_pass * grad_bytes + 2 * one_pass * param_bytes  # RS(grads) + 2 x AG(weights)


def warmup_decay_lr(t, min_lr, max_lr, warmup_steps, total_steps):
    """Learning rate of optimizer step t (t >= 1): the piecewise-linear curve
    through (0, min_lr), (warmup_steps, max_lr), (total_steps, 0), flat at 0
    beyond, read at k = t - 1 schedule steps; rounded once to float32."""
    if t < 1 or warmup_steps < 0 or total_steps <= warmup_steps:
        raise ValueError("need t >= 1 and 0 <= warmup_steps < total_steps")
    k = t - 1
    if k < warmup_steps:
        frac = k / warmup_steps
        lr = min_lr + frac * (max_lr - min_lr)
    elif k < total_steps:
        frac = (k - warmup_steps) / (total_steps - warmup_steps)
        lr = max_lr - frac * max_lr
    else:
        lr = 0.0
    return float(np.float32(lr))
