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
    assert cfg.ignored == ["train_micro_batch_size_per_gpu", "zero_optimization.contiguous_gradients",
                           "zero_optimization.overlap_comm"]


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
