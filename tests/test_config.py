"""The configuration subset the engines read (no GPU): keys, defaults, refusals."""
import pytest

from zero_sharded_mixed_gb300.config import ZeroConfig


def test_reads_the_keys_of_a_deepspeed_configuration():
    cfg = ZeroConfig.from_dict({
        "train_micro_batch_size_per_gpu": 4,
        "gradient_accumulation_steps": 8,
        "gradient_clipping": 1.0,
        "bf16": {"enabled": True},
        "optimizer": {"type": "AdamW", "params": {"lr": 3e-4, "betas": [0.9, 0.95], "eps": 1e-8,
                                                  "weight_decay": 0.1}},
        "zero_optimization": {"stage": 2, "reduce_bucket_size": 2e8, "overlap_comm": True,
                              "contiguous_gradients": True},
    })
    assert (cfg.stage, cfg.reduce_bucket_size, cfg.gradient_accumulation_steps) == (2, 200_000_000, 8)
    assert (cfg.gradient_clipping, cfg.lr, cfg.betas, cfg.eps, cfg.weight_decay) == (1.0, 3e-4, (0.9, 0.95),
                                                                                    1e-8, 0.1)
    assert not cfg.zero_quantized_weights and not cfg.zero_quantized_gradients
    assert cfg.ignored == ["train_micro_batch_size_per_gpu", "zero_optimization.contiguous_gradients"]
    assert cfg.overlap_comm


def test_defaults_and_zeropp_switches():
    cfg = ZeroConfig.from_dict({})
    assert (cfg.stage, cfg.reduce_bucket_size, cfg.gradient_accumulation_steps, cfg.gradient_clipping) == \
        (2, 500_000_000, 1, 0.0)
    cfg = ZeroConfig.from_dict({"zero_optimization": {"stage": 3, "zero_quantized_weights": True,
                                                      "zero_quantized_gradients": True}})
    assert cfg.stage == 3 and cfg.zero_quantized_weights and cfg.zero_quantized_gradients


@pytest.mark.parametrize("bad", [
    {"zero_optimization": {"stage": 0}},
    {"zero_optimization": {"stage": 4}},
    {"zero_optimization": {"stage": 2, "zero_quantized_weights": True}},
    {"zero_optimization": {"offload_optimizer": {"device": "cpu"}}},
    {"zero_optimization": {"stage": 3, "offload_param": {"device": "nvme"}}},
    {"fp16": {"enabled": True}},
    {"bf16": {"enabled": False}},
    {"optimizer": {"type": "SGD", "params": {"lr": 0.1}}},
    {"gradient_accumulation_steps": 0},
    {"gradient_clipping": -1.0},
    {"optimizer": {"type": "AdamW", "params": {"betas": [1.0, 0.999]}}},
])
def test_refuses_what_the_build_does_not_do(bad):
    with pytest.raises(ValueError):
        ZeroConfig.from_dict(bad)


def test_offload_to_none_is_accepted():
    cfg = ZeroConfig.from_dict({"zero_optimization": {"stage": 3, "offload_param": {"device": "none"}}})
    assert cfg.stage == 3


def test_the_pages_example_configuration_with_its_scheduler():
    """"DeepSpeed ZeRO", "The configuration file", as printed."""
    cfg = ZeroConfig.from_dict({
        "train_micro_batch_size_per_gpu": 4,
        "gradient_accumulation_steps": 8,
        "bf16": {"enabled": True},
        "zero_optimization": {"stage": 2, "overlap_comm": True, "contiguous_gradients": True,
                              "reduce_bucket_size": 200000000, "allgather_bucket_size": 200000000},
        "gradient_clipping": 1.0,
        "optimizer": {"type": "AdamW", "params": {"lr": 0.0001, "betas": [0.9, 0.999], "weight_decay": 0.01}},
        "scheduler": {"type": "WarmupDecayLR",
                      "params": {"warmup_min_lr": 0, "warmup_max_lr": 0.0001, "warmup_num_steps": 100,
                                 "total_num_steps": 10000}},
    })
    assert cfg.scheduler == {"min_lr": 0.0, "max_lr": 1e-4, "warmup_steps": 100, "total_steps": 10000}
    assert "scheduler" not in cfg.ignored
    assert (cfg.stage, cfg.reduce_bucket_size, cfg.gradient_accumulation_steps) == (2, 200_000_000, 8)


@pytest.mark.parametrize("sched", [
    {"type": "OneCycle", "params": {}},
    {"type": "WarmupDecayLR", "params": {"warmup_num_steps": 10}},
    {"type": "WarmupDecayLR", "params": {"warmup_num_steps": 10, "total_num_steps": 10}},
    {"type": "WarmupDecayLR", "params": {"warmup_num_steps": 10, "total_num_steps": 20, "warmup_type": "log"}},
    {"type": "WarmupDecayLR", "params": {"warmup_num_steps": 10, "total_num_steps": 20, "warmup_min_lr": -1}},
])
def test_refuses_schedulers_it_does_not_implement(sched):
    with pytest.raises(ValueError):
        ZeroConfig.from_dict({"scheduler": sched})


def test_the_library_schedule_matches_the_oracle(zlib):
    """lr_at (the library's zero_lr_warmup_decay) against the oracle's restatement,
    within one float32 ulp at every step of two schedules, exactly at the knots."""
    import numpy as np

    from oracle import formulas
    for sp in ({"warmup_min_lr": 0, "warmup_max_lr": 1e-4, "warmup_num_steps": 100, "total_num_steps": 10000},
               {"warmup_min_lr": 3e-6, "warmup_max_lr": 6e-4, "warmup_num_steps": 0, "total_num_steps": 777}):
        cfg = ZeroConfig.from_dict({"scheduler": {"type": "WarmupDecayLR", "params": sp}})
        sc = cfg.scheduler
        ts = np.arange(1, sc["total_steps"] + 50)
        got = np.array([cfg.lr_at(int(t)) for t in ts], np.float32)
        ref = np.array([formulas.warmup_decay_lr(int(t), sc["min_lr"], sc["max_lr"], sc["warmup_steps"],
                                                 sc["total_steps"]) for t in ts], np.float32)
        ulps = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
        assert ulps.max() <= 1
        for t in (1, sc["warmup_steps"] + 1, sc["total_steps"] + 1):
            assert got[t - 1] == ref[t - 1]
    assert ZeroConfig.from_dict({}).lr_at(5) == 1e-4                        # no scheduler: the optimizer's lr
    with pytest.raises(zlib.ZeroError):
        zlib.zero_lr_warmup_decay(0, 0.0, 1e-4, 10, 20)
