"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the optimizer step: it only draws random
numbers and lists tensor shapes.  Both the CUDA path and the oracle are fed
from it; neither computes anything here.

Shapes follow the models the pages use as examples (GPT-2 XL, the 1.5B model of
"ZeRO: How DeepSpeed Made Trillion-Parameter Training Practical", section
"Where the 16 bytes per parameter comes from"; a 7B decoder of "ZeRO Optimizer,
in depth", "Worked example: a 7B model on eight 80 GB GPUs"), with the
architectures' published dimensions:

* GPT-2 XL: 48 blocks, d = 1600, ffn = 6400, vocab 50257, 1024 positions, head
  tied to the token embedding -> N = 1,557,611,200.
* Llama-7B: 32 blocks, d = 4096, ffn = 11008, vocab 32000, untied head
  -> N = 6,738,415,616.

Value distributions: fp32 master weights ~ Normal(0, 0.02); bf16 gradients
drawn as fp32 ~ Normal(0, 1e-3), optionally with a Bernoulli(p) mask of
outliers scaled by 100, then rounded to bf16 by torch; Adam moments start at
zero.  The padding tail of every flat buffer is zero.
"""
from __future__ import annotations

import torch

# --------------------------------------------------------------------------
# model shapes (per-tensor element counts, in flattening order)
# --------------------------------------------------------------------------


def gpt2xl_numels(n_layer: int = 48, d: int = 1600, ffn: int = 6400,
                  vocab: int = 50257, n_ctx: int = 1024) -> list[int]:
    out = [vocab * d, n_ctx * d]                        # wte (tied head), wpe
    for _ in range(n_layer):
        out += [d, d,                                   # ln_1 weight, bias
                d * 3 * d, 3 * d,                       # attn qkv weight, bias
                d * d, d,                               # attn proj weight, bias
                d, d,                                   # ln_2 weight, bias
                d * ffn, ffn,                           # mlp fc weight, bias
                ffn * d, d]                             # mlp proj weight, bias
    out += [d, d]                                       # ln_f weight, bias
    return out


def llama7b_block_numels(d: int = 4096, ffn: int = 11008) -> list[int]:
    return [d,                                          # input norm
            d * d, d * d, d * d, d * d,                 # q, k, v, o
            d,                                          # post-attention norm
            ffn * d, ffn * d, d * ffn]                  # gate, up, down


def llama7b_units(n_layer: int = 32, d: int = 4096, ffn: int = 11008,
                  vocab: int = 32000) -> list[list[int]]:
    """ZeRO-3 units: the embedding, one unit per block, then final norm + head."""
    units = [[vocab * d]]
    units += [llama7b_block_numels(d, ffn) for _ in range(n_layer)]
    units.append([d, vocab * d])
    return units


def llama7b_numels(**kw) -> list[int]:
    return [x for unit in llama7b_units(**kw) for x in unit]


# --------------------------------------------------------------------------
# seeded generators
# --------------------------------------------------------------------------


def derive_seed(seed: int, *parts: int) -> int:
    """A fixed, documented mixing of (seed, step, rank, micro-batch, ...)."""
    s = int(seed) & 0xFFFFFFFF
    for p in parts:
        s = (s * 1_000_003 + int(p) + 0x9E37) & 0x7FFFFFFFFFFF
    return s


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def master_weights(n_real: int, padded: int, seed: int = 0, device="cpu",
                   std: float = 0.02) -> torch.Tensor:
    """fp32 flat master weights, Normal(0, std) on [0, n_real), zero padding."""
    out = torch.zeros(padded, dtype=torch.float32, device=device)
    if n_real:
        out[:n_real].normal_(0.0, std, generator=_gen(device, derive_seed(seed, 1)))
    return out


def grad_bf16_into(out: torch.Tensor, n_real: int, seed: int, step: int, rank: int,
                   micro: int = 0, std: float = 1e-3, outlier_p: float = 0.0,
                   outlier_scale: float = 100.0, chunk: int = 1 << 28) -> torch.Tensor:
    """Fill ``out`` (bf16, flat, padded) with one rank's gradient for one step.

    Drawn in fp32 chunks so that large vectors need little temporary memory;
    rounded to bf16 by torch.  The tail past ``n_real`` is zero.
    """
    assert out.dtype == torch.bfloat16 and out.dim() == 1
    dev = out.device
    g = _gen(dev, derive_seed(seed, 2, step, rank, micro))
    out[n_real:].zero_()
    for lo in range(0, n_real, chunk):
        hi = min(n_real, lo + chunk)
        x = torch.empty(hi - lo, dtype=torch.float32, device=dev)
        x.normal_(0.0, std, generator=g)
        if outlier_p > 0.0:
            mask = torch.empty(hi - lo, dtype=torch.float32, device=dev)
            mask.uniform_(0.0, 1.0, generator=g)
            x = torch.where(mask < outlier_p, x * outlier_scale, x)
        out[lo:hi].copy_(x)
    return out


def grads_bf16(n_dp: int, n_real: int, padded: int, seed: int, step: int, device="cpu",
               micro: int = 0, **kw) -> torch.Tensor:
    """(n_dp, padded) bf16: row r is simulated rank r's full local gradient."""
    out = torch.empty((n_dp, padded), dtype=torch.bfloat16, device=device)
    for r in range(n_dp):
        grad_bf16_into(out[r], n_real, seed, step, r, micro, **kw)
    return out


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


def from_bf16_bits(a, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    import numpy as np
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
