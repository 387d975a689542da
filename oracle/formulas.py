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
"""
from __future__ import annotations


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
