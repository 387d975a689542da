"""The benchmark's command line and the reference arm's JSON line (CPU only)."""
import io
import json
from contextlib import redirect_stdout

import pytest

import bench


def test_defaults():
    a = bench.parse_args([])
    assert (a.gpus, a.impl, a.workload) == (1, "ours", "gpt2xl")
    assert a.warmup >= 3 and a.steps >= 1


def test_reference_arm_line(monkeypatch):
    monkeypatch.setattr(bench, "REF_SAMPLE", 1 << 12)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


def test_reference_arm_other_ranks_are_silent(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert buf.getvalue() == ""


def test_owner_count_of_a_range():
    """The 8-bit gradient kernels launch once per owner a range meets, or once
    for a range of several whole shards."""
    import bench

    class L:
        shard = 100
    assert bench._owners(L, 0, 100) == 1
    assert bench._owners(L, 0, 101) == 2
    assert bench._owners(L, 99, 201) == 3
    assert bench._owners(L, 150, 150) == 0
    assert bench._owners(L, 0, 800) == 1
    assert bench._owners(L, 200, 500) == 1
    assert bench._owners(L, 200, 550) == 4

    class L8:
        shard = 96
    assert bench._owners(L8, 0, 150) == 1          # one stream over owners 0 and 1
    assert bench._owners(L8, 8, 500) == 1
    assert bench._owners(L8, 4, 150) == 2          # off the 8-element grid: one launch per owner
    assert bench._owners(L8, 100, 150) == 1


@pytest.mark.parametrize("name", ["gpt2xl", "llama7b-shard", "gpt2xl-clip", "gpt2xl-qgrad", "accum-zero1",
                                  "accum-zero2", "zero3", "zero3-fused", "zero3-fused-graph", "zero3-prefetch",
                                  "zero3-int8", "zero3-int8-fused", "zero3-zeropp", "zero3-zeropp-fused",
                                  "zero3-compute", "zero3-prefetch-compute"])
def test_every_workload_has_an_oracle_step(name):
    """The bench times the oracle beside every workload: its statement of the
    step runs on a small sample and moves the weights."""
    import numpy as np

    import bench
    step, n, what = bench.oracle_workload_step(name, 4096)
    assert n == 4096 and "owned elements" in what
    cells = step.__closure__
    step(1)
    step(2)
    st = next(c.cell_contents for c in cells if isinstance(c.cell_contents, dict) and "w" in c.cell_contents)
    assert np.isfinite(st["w"]).all() and (st["m"] != 0).any()


def test_threaded_oracle_timing_covers_the_sample():
    """The all-cores CPU baseline steps every chunk of the sample."""
    import numpy as np

    from zero_sharded_mixed_gb300 import inputs
    n, n_dp = 10_000, 4
    g = inputs.bf16_bits(inputs.grads_bf16(n_dp, n, n, seed=1, step=1))
    sample = (g, inputs.master_weights(n, n, seed=1).numpy(), np.zeros(n, np.float32), np.zeros(n, np.float32))
    rate, secs, done = bench.time_oracle(sample, 0.2, n_dp, threads=3)
    assert rate > 0 and secs >= 0.2 and done >= n


def _fake_result(workload, value, ms, frac):
    roof = {"bound": "hbm", "achieved": frac * 6675.2, "peak": 6675.2, "unit": "GB/s", "frac": frac,
            "peak_kind": "measured", "traffic": 42.02 * 194701400, "algorithmic_bytes_per_launch": 21e9,
            "kernel": "rs_adamw", "kernel_symbols": "zgb::rs_adamw_vec_kernel<0,8> (bf16 sources x 8)"}
    return {
        "value": value, "ms_per_step": ms, "steps": 20, "step_ms_median": ms, "step_ms_min": ms * 0.99,
        "hbm_gbs_step": 7000.0, "bytes_per_param_step": 42,
        "config": {"workload": workload, "model": "GPT-2-XL shapes", "N": 1557611200, "n_dp": 8,
                   "shard": 194701400, "padded_n": 1557611200, "bucket": 500000000, "buckets": 4,
                   "l2": "inputs 50.0 GB > 129 MB L2, no flush"},
        "roofline": roof,
        "kernels": {"rs_adamw": {"launches_per_step": 4, "ms_per_step": ms, "bytes_per_step": 65419670400,
                                 "achieved_gbs": 7000.0}},
        "gpu_launches": 80,
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "power_w_max": 1086.5, "samples": 40,
                   "reasons": []},
        "e2e": {"value": 1.2e10, "unit": bench.UNIT, "ms_per_step": 130.0, "steps": 10, "step_ms_min": 124.8,
                "step_ms_median": 126.0,
                "h2d_bytes_per_step": 24921779200, "d2h_bytes_per_step": 3115222400,
                "link": {"h2d_gbs": 190.0, "h2d_ms_per_step": 124.0, "frac": 0.95}},
        "cpu_baseline": {"value": 1.4e9, "unit": bench.UNIT, "cores": 16, "kind": "oracle",
                         "single_core_value": 9e7,
                         "sample": "first 33554432 owned elements (all 8 gradient slices), 16 chunks, one "
                                   "thread each; 12.3 passes in 6.0 s"},
    }


def test_headline_line_is_compact_and_parses():
    """The headline line carries every key of the contract, parses as JSON on
    its own and stays under 2 KB, so that a short tail of the log holds it."""
    args = bench.parse_args(["--steps", "20", "--warmup", "5"])
    p = _fake_result("gpt2xl_zero2_all_shards", 1.68e11, 9.26, 1.06)
    seven = bench.target_7b(dict(_fake_result("llama7b_zero2_one_shard", 2.0e11, 4.2, 1.04)))
    line = bench.headline_line(p, args, 1, seven)
    text = json.dumps(line)
    assert len(text) < 2048
    back = json.loads(text)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "clocks", "gpu_launches", "impl", "target_7b"):
        assert key in back, key
    assert back["config"]["workload"] == "gpt2xl_zero2_all_shards" and back["value"] > 0
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in back["roofline"], key
    assert back["e2e"]["h2d_bytes_per_step"] > 0 and back["e2e"]["d2h_bytes_per_step"] > 0
    assert back["target_7b"]["frac"] == 1.04 and back["target_7b"]["met"] is True
    assert back["target_7b"]["frac_nominal"] == pytest.approx(1.04 * 6675.2 / bench.NOMINAL_HBM_GBS)
    assert back["cpu_baseline"]["cores"] == 16 and back["impl"] == "ours"


def test_headline_line_stays_short_with_long_fields():
    """Long optional fields are dropped before the line passes the limit."""
    args = bench.parse_args([])
    p = _fake_result("gpt2xl_zero2_all_shards", 1.68e11, 9.26, 1.06)
    p["cpu_baseline"]["sample"] = "x" * 3000
    line = bench.headline_line(p, args, 1, None)
    assert len(json.dumps(line)) <= bench.HEADLINE_MAX_CHARS
    assert line["value"] == p["value"] and line["cpu_baseline"]["value"] == p["cpu_baseline"]["value"]


def test_workload_lines_carry_no_headline_keys():
    """The lines of the other workloads cannot be taken for the headline."""
    line = bench.workload_line("llama7b-shard", _fake_result("llama7b_zero2_one_shard", 2e11, 4.2, 1.04))
    assert "metric" not in line and "value" not in line
    assert line["workload_result"] == "llama7b-shard" and line["params_per_s"] == 2e11
    json.loads(json.dumps(line))


def test_default_run_has_no_stand_in_matmuls():
    """The workloads with cuBLAS stand-in layer compute run only on request."""
    order = bench.workload_order(bench.parse_args([]))
    assert order[0] == "gpt2xl" and "llama7b-shard" in order
    assert not set(bench.COMPUTE_WORKLOADS) & set(order)
    assert set(bench.COMPUTE_WORKLOADS) <= set(bench.workload_order(bench.parse_args(["--with-compute"])))
    assert bench.workload_order(bench.parse_args(["--no-extra"])) == ["gpt2xl"]
    assert bench.workload_order(bench.parse_args(["--workload", "probe"])) == ["probe"]


def test_cast_workload_oracle_step_and_order():
    """The cast workload is a default extra workload, and the oracle's
    statement of it casts the sample's master weights."""
    assert "cast" in bench.workload_order(bench.parse_args([]))
    step, n, what = bench.oracle_workload_step("cast", 4096)
    assert n == 4096 and "owned elements" in what and "cast" in what
    step(1)


def test_e2e_host_bytes_with_a_shared_row():
    """The e2e fallback pins one gradient row instead of one per rank."""
    import torch

    class W:
        grads = torch.empty((8, 1000), dtype=torch.bfloat16)
        out = torch.empty(1000, dtype=torch.bfloat16)
    assert bench.e2e_host_bytes(W) == 8 * 1000 * 2 + 1000 * 2
    assert bench.e2e_host_bytes(W, shared_rows=True) == 1000 * 2 + 1000 * 2


def test_printed_floats_keep_six_significant_digits():
    r = bench._rounded({"a": 168211715564.56232, "b": [1.0595268135262763, 3], "c": {"d": 0.000123456789}})
    assert r == {"a": 168212000000.0, "b": [1.05953, 3], "c": {"d": 0.000123457}}
