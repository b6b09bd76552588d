"""The seeded workload recipes: shapes, dtypes, determinism and the
distribution facts the recipes promise."""

import torch

from log_linear_attention_chunkwise_gb300 import workloads as W


def test_levels_per_workload():
    assert [c.L for c in W.FWD_CONFIGS.values()] == [9, 12, 14, 16]


def test_small_workload_shapes_and_determinism():
    cfg = W.FWD_CONFIGS["fp32_T256"]
    a = W.make_fwd_inputs(cfg)
    b = W.make_fwd_inputs(cfg)
    assert a["q"].shape == (1, 2, 256, 32) and a["q"].dtype == torch.float32
    assert a["lam"].shape == (1, 2, 256, 9)
    for n in a:
        assert torch.equal(a[n], b[n])
    assert (a["g"] <= 0).all() and (a["lam"] >= 0).all()
    norms = a["k"].norm(dim=-1)
    assert torch.allclose(norms, torch.ones_like(norms), atol=1e-5)


def test_bf16_rounding_and_lambda_one_mask():
    cfg = W.FWD_CONFIGS["bf16_T8192_lam1"].with_(B=1, T=256)
    x = W.make_fwd_inputs(cfg)
    assert x["q"].dtype == torch.bfloat16 and x["g"].dtype == torch.float32
    is_one = (x["lam"] == 1.0).all(dim=2)[0]  # [H, L]
    frac = is_one.float().mean().item()
    assert 0.3 < frac < 0.7
    # the mask is shared over tokens: a pair is either all ones or none
    anyone = (x["lam"] == 1.0).any(dim=2)[0]
    assert torch.equal(anyone, is_one)


def test_slow_decay_recipe_mean_gate():
    cfg = W.FWD_CONFIGS["bf16_T32768_slowdecay"].with_(T=4096, H=2)
    g = W.make_fwd_inputs(cfg)["g"]
    assert -0.22 < g.mean().item() < -0.15  # E[-softplus(N(-2,1))] is about -0.18


def test_decode_positions_range():
    cfg = W.DECODE_CONFIG
    pos = W.make_decode_positions(cfg)
    assert pos.shape == (64,) and pos.min() >= 1 and pos.max() <= 65536
    # after all steps the state never needs more than Ls = 17 slots
    assert int(pos.max() + cfg.steps).bit_length() <= cfg.Ls
