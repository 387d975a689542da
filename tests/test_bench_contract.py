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
