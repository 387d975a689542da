"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source, on the CPU:
a dropped term, a wrong sign, index, operand or constant, a rounding rule
changed.  The copy is compiled, swapped in for the real oracle, and the pins
of tests/test_oracle_*.py are run against it.  At least one must fail, or the
pins would not have noticed that mistake.  Every planted mistake stays inside
the arrays' bounds."""
import ctypes
import os
import subprocess

import numpy as np

import pytest

import oracle
from tests import test_oracle_cast as pc
from tests import test_oracle_clip as pk
from tests import test_oracle_layout as pl
from tests import test_oracle_qgrad as pg
from tests import test_oracle_quant as pq
from tests import test_oracle_step as ps

SRC = os.path.join(os.path.dirname(oracle.__file__), "zero_oracle.c")

# (what, exact text in the oracle, the mistake)
MUTATIONS = [
    ("bias correction of m dropped", "float m_hat = mi / bc1;", "float m_hat = mi;"),
    ("Adam step with the wrong sign", "wi = wi - lr * (m_hat", "wi = wi + lr * (m_hat"),
    ("eps inside the square root", "(sqrtf(v_hat) + eps)", "sqrtf(v_hat + eps)"),
    ("weight decay dropped", "wi = wi - lr_wd * wi;", ";"),
    ("beta1 used for v", "float vi = b2 * v[i]", "float vi = b1 * v[i]"),
    ("gradient not squared in v", "one_minus_b2 * (gi * gi)", "one_minus_b2 * gi"),
    ("bias-correction exponent off by one", "*bc1 = (float)(1.0 - pow((double)b1, (double)t));",
     "*bc1 = (float)(1.0 - pow((double)b1, (double)(t + 1)));"),
    ("mean divides by n_dp + 1", "shard,\n                                (float)n_dp, g);",
     "shard,\n                                (float)(n_dp + 1), g);"),
    ("rank reads the next rank's shard", "oracle_reduce_mean_bf16(grads + (int64_t)o * shard,",
     "oracle_reduce_mean_bf16(grads + (int64_t)((o + 1) % n_dp) * shard,"),
    ("sources summed in reverse order",
     "s = s + src[(int64_t)r * ld + i];\n        g[i] = s / divisor;",
     "s = s + src[(int64_t)(n_src - 1 - r) * ld + i];\n        g[i] = s / divisor;"),
    ("bf16 ties rounded away from zero", "if (kept & 1u) kept += 1u;", "kept += 1u;"),
    ("bf16 cast truncates", "if (dropped > 0x8000u) {", "if (dropped > 0xffffu) {"),
    ("bf16 cast makes every NaN the canonical one", "return (uint16_t)((u >> 16) | 0x0040u);",
     "return (uint16_t)((u >> 16 & 0x8000u) | 0x7fc0u);"),
    ("shard length not rounded up to the alignment", "if (shard * align < per_rank) shard += 1;", ";"),
    ("shard length floors N / n_dp", "if (per_rank * n_dp < total) per_rank += 1;", ";"),
    ("accumulation ignores the first flag", "acc[i] = first ? x : acc[i] + x;", "acc[i] = acc[i] + x;"),
    ("gather concatenates in reverse rank order",
     "full[(int64_t)o * shard + i] = shards[(int64_t)o * shard + i];",
     "full[(int64_t)o * shard + i] = shards[(int64_t)(n_dp - 1 - o) * shard + i];"),
    ("clip divides by the squared norm", "(sqrt(norm_sq) + 1e-6)", "(norm_sq + 1e-6)"),
    ("clip coefficient not capped at 1", "return c < 1.0f ? c : 1.0f;", "return c;"),
    ("norm sum drops its compensation", "return k->sum + k->comp;", "return k->sum;"),
    ("norm sum adds each square twice", "oracle_csum_add(&acc, g * g);\n    }\n    return oracle_csum_value(&acc);\n}\n\nfloat",
     "oracle_csum_add(&acc, g * g);\n        oracle_csum_add(&acc, g * g);\n    }\n    return oracle_csum_value(&acc);\n}\n\nfloat"),
    ("8-bit scale uses 126", "float inv = 127.0f / amax;", "float inv = 126.0f / amax;"),
    ("8-bit codes truncated", "nearbyintf(oracle_bf16_to_f32(w[i]) * inv)",
     "truncf(oracle_bf16_to_f32(w[i]) * inv)"),
    ("8-bit dequantization uses the first block's scale", "scales[i / block]", "scales[0]"),
    ("8-bit gradient uses the previous block's scale", "block_scales[k / block];",
     "block_scales[k / block > 0 ? k / block - 1 : 0];"),
    ("8-bit gradient rounded to bf16 before the mean",
     "out[k] = (float)codes[k] * block_scales[k / block];",
     "out[k] = oracle_bf16_to_f32(oracle_f32_to_bf16((float)codes[k] * block_scales[k / block]));"),
    ("8-bit gradient loses the code's sign", "out[k] = (float)codes[k] *", "out[k] = fabsf((float)codes[k]) *"),
]


def _pins():
    """The pins, as (name, callable) -- parametrized ones with representative
    arguments."""
    return [
        ("torch AdamW", ps.test_single_rank_matches_torch_adamw),
        ("first-step closed form", ps.test_first_step_closed_form),
        ("constant-gradient closed form", ps.test_constant_gradient_closed_form),
        ("zero gradient", ps.test_zero_gradient_is_pure_decay),
        ("bias corrections", ps.test_bias_corrections),
        ("DP equivalence", lambda: ps.test_zero_step_equals_data_parallel(4, 4096, 8)),
        ("DP equivalence ragged", lambda: ps.test_zero_step_equals_data_parallel(3, 1000, 1)),
        ("shard gets its piece", ps.test_zero_step_shard_gets_its_own_gradient_piece),
        ("dyadic mean", lambda: ps.test_mean_is_exact_for_dyadic_power_of_two(4)),
        ("one rounding of the sum", lambda: ps.test_mean_is_one_rounding_of_exact_sum(3)),
        ("summation order", ps.test_mean_fp32_rows_and_order),
        ("accumulation orders", ps.test_accumulation_orders_agree_exactly_on_dyadic_inputs),
        ("single micro-batch", ps.test_single_micro_batch_accumulation_is_the_mean),
        ("first micro-batch overwrites", ps.test_first_micro_batch_overwrites_the_buffer),
        ("gather", ps.test_all_gather_is_concatenation),
        ("cast specials", pc.test_special_values),
        ("cast low halves", pc.test_every_low_half_for_some_upper_halves),
        ("cast NaN round trip", pc.test_quiet_nan_payload_survives_a_widening_round_trip),
        ("layout brute force", lambda: pl.test_brute_force_small(8)),
        ("workload layouts", pl.test_workload_layouts),
        ("clip vs torch", lambda: pk.test_clip_matches_torch(1.0, 1.0)),
        ("clip closed forms", pk.test_closed_forms),
        ("norm vs numpy", pk.test_norm_matches_numpy_fp64),
        ("norm vs exact sum", pk.test_norm_is_the_exact_sum_of_squares),
        ("quant error bound", lambda: pq.test_roundtrip_error_bound(256, 4097)),
        ("quant max and symmetry", pq.test_block_max_maps_to_127_and_symmetry),
        ("quant ties and zeros", pq.test_ties_to_even_and_zero_blocks),
        ("quant ragged", pq.test_ragged_last_block_and_wire_bytes),
        ("8-bit gradient exact codes",
         lambda: pg.test_exact_gradients_quantize_to_their_codes_and_step_like_bf16(4, 1000, 256)),
        ("8-bit gradient error bound", lambda: pg.test_error_within_half_a_step(4, 5000, 256)),
        ("8-bit gradient slices", pg.test_blocks_restart_at_every_slice),
        ("8-bit gradient accumulation", pg.test_exact_gradients_accumulate_like_bf16),
        ("8-bit first micro-batch overwrites", pg.test_first_micro_batch_overwrites_the_buffer),
    ]


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_a_planted_mistake_fails_a_pin(what, old, new, tmp_path, monkeypatch):
    src = open(SRC).read()
    assert src.count(old) == 1, f"the mutation target for '{what}' must occur exactly once"
    mutated = tmp_path / "mutated.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmutated.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", str(so), str(mutated), "-lm"])
    lib = oracle.configure(ctypes.CDLL(str(so)))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for name, pin in _pins():
        try:
            pin()
        except (Exception, pytest.fail.Exception):   # an assertion, a failed pytest.raises, a ValueError
            caught.append(name)
    assert caught, f"no pin noticed: {what}"


def test_the_real_oracle_passes_every_pin():
    for name, pin in _pins():
        pin()


# Mistakes in the oracle's Python composition of the C routines (the 8-bit
# gradient functions slice, offset and combine them).  Each mutant replaces one
# function of the oracle module.

def _q_whole_rows(g_rows, n_dp, block=256):
    """Blocks that do not restart at slice boundaries: each row quantized whole."""
    g = oracle._u16(g_rows)
    n_src, P = g.shape
    S = P // n_dp
    nb = -(-S // block)
    q = np.empty((n_src, P), dtype=np.int8)
    scales = np.zeros((n_src, n_dp * nb), dtype=np.float32)
    for r in range(n_src):
        q[r], s = oracle.quantize_int8(g[r], block)
        scales[r, :s.size] = s[:n_dp * nb]
    return q, scales


def _deq_first_slice_scales(q_rows, scale_rows, n_dp, block=256):
    """Every slice dequantized with slice 0's scales."""
    q = np.ascontiguousarray(q_rows, dtype=np.int8)
    sc = oracle._f32(scale_rows)
    n_src, P = q.shape
    S = P // n_dp
    nb = -(-S // block)
    out = np.empty((n_src, P), dtype=np.float32)
    for r in range(n_src):
        for o in range(n_dp):
            k = np.arange(S)
            out[r, o * S:(o + 1) * S] = q[r, o * S:(o + 1) * S].astype(np.float32) * sc[r, k // block]
    return out


def _acc_int8_ignores_first(acc, q_rows, scale_rows, n_dp, block, first):
    x = oracle.reduce_mean(oracle.dequantize_grad_int8(q_rows, scale_rows, n_dp, block), 1.0)
    return x if acc is None else (oracle._f32(acc) + x).astype(np.float32)


def _qgrad_ref_wrong_divisor(q_rows, scale_rows, n_dp, block, divisor, w, m, v, hp, t):
    g = oracle.reduce_mean(oracle.dequantize_grad_int8(q_rows, scale_rows, n_dp, block), divisor * 2)
    w2, m2, v2 = oracle.adamw(w, m, v, g, hp, t)
    return oracle.cast_bf16(w2), w2, m2, v2


PY_MUTATIONS = [
    ("8-bit gradient blocks do not restart at slices", "quantize_grad_int8", _q_whole_rows),
    ("8-bit gradient slices use slice 0's scales", "dequantize_grad_int8", _deq_first_slice_scales),
    ("8-bit accumulation ignores the first flag", "accumulate_reduce_int8", _acc_int8_ignores_first),
    ("8-bit step divides twice", "qgrad_rs_adamw_reference", _qgrad_ref_wrong_divisor),
]


@pytest.mark.parametrize("what,name,fn", PY_MUTATIONS, ids=[m[0] for m in PY_MUTATIONS])
def test_a_planted_composition_mistake_fails_a_pin(what, name, fn, monkeypatch):
    monkeypatch.setattr(oracle, name, fn)
    caught = []
    for pin_name, pin in _pins():
        try:
            pin()
        except (Exception, pytest.fail.Exception):
            caught.append(pin_name)
    assert caught, f"no pin noticed: {what}"


# Mistakes in the memory, communication and schedule formulas (oracle/formulas.py):
# each mutant is loaded as a module in place of the real one, and the pins of
# tests/test_oracle_formulas.py (the pages' printed numbers, the ring factor,
# the invalid-stage rule) run against it.
FORMULA_SRC = os.path.join(os.path.dirname(oracle.__file__), "formulas.py")
FORMULA_MUTATIONS = [
    ("stage 2 keeps the full gradients", "grads = grads / n_dp ", "grads = grads * 1 "),
    ("stage 1 shards the optimizer over n_dp - 1", "optimizer = optimizer / n_dp ",
     "optimizer = optimizer / (n_dp - 1) "),
    ("stage 3 keeps the full weights", "weights = weights / n_dp ", "weights = weights * 1 "),
    ("16 bytes per parameter become 18", "weights = 2 * N", "weights = 4 * N"),
    ("ring factor dropped", "one_pass = (n_dp - 1) / n_dp * N", "one_pass = N"),
    ("stage 3 gathers the weights once", "return one_pass * grad_bytes + 2 * one_pass * param_bytes",
     "return one_pass * grad_bytes + one_pass * param_bytes"),
    ("stage 0 reduce-scatters only", "return 2 * one_pass * grad_bytes", "return one_pass * grad_bytes"),
    ("stage 4 accepted", "if stage not in (0, 1, 2, 3):\n        raise ValueError(f\"ZeRO stage must be 0, 1, 2 or 3, got {stage!r}\")\n    weights",
     "if stage not in (0, 1, 2, 3, 4):\n        raise ValueError(f\"ZeRO stage must be 0, 1, 2 or 3, got {stage!r}\")\n    weights"),
    ("schedule read at step t instead of t - 1", "    k = t - 1\n", "    k = t\n"),
    ("decay ends at the minimum", "lr = max_lr - frac * max_lr", "lr = max_lr - frac * (max_lr - min_lr)"),
    ("warmup runs down from the maximum", "lr = min_lr + frac * (max_lr - min_lr)",
     "lr = max_lr - frac * (max_lr - min_lr)"),
    ("the maximum kept after total_num_steps", "        lr = 0.0", "        lr = max_lr"),
]


@pytest.mark.parametrize("what,old,new", FORMULA_MUTATIONS, ids=[m[0] for m in FORMULA_MUTATIONS])
def test_a_planted_formula_mistake_fails_a_pin(what, old, new, monkeypatch):
    import importlib.util
    import types

    from tests import test_oracle_formulas as pf
    src = open(FORMULA_SRC).read()
    assert src.count(old) == 1, f"the mutation target for '{what}' must occur exactly once"
    mutant = types.ModuleType("formulas_mutant")
    exec(compile(src.replace(old, new), "formulas_mutant", "exec"), mutant.__dict__)
    monkeypatch.setattr(pf, "formulas", mutant)
    pins = [lambda c=c: pf.test_memory_matches_printed_numbers(c) for c in pf._golden()["memory"]]
    pins += [pf.test_free_memory_after_states, pf.test_sixteen_bytes_per_parameter,
             pf.test_per_gpu_formulas_are_the_table, pf.test_stage_limits,
             pf.test_comm_stage12_equals_dp_and_stage3_is_one_and_a_half, pf.test_comm_exact_ring_factor,
             pf.test_comm_fp32_gradients_double_the_gradient_term, pf.test_comm_llama3_70b_printed]
    pins += [lambda s=s: pf.test_invalid_stage_raises(s) for s in (-1, 4, 5, "1", None, 1.5)]
    pins += [pf.test_schedule_points_of_the_example_configuration, pf.test_schedule_is_linear_in_each_phase,
             pf.test_schedule_with_a_minimum_and_without_warmup]
    caught = 0
    for pin in pins:
        try:
            pin()
        except (Exception, pytest.fail.Exception):
            caught += 1
    assert caught, f"no pin noticed: {what}"
