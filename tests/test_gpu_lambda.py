"""GPU parity of lla_lambda_mlp (the level-weight producer of "Adaptive memory
decay for Log-Linear Attention") against the fp64 oracle, and its use as the
forward's lambda."""

import math

import numpy as np
import pytest
import torch

import oracle
from log_linear_attention_chunkwise_gb300 import binding
from log_linear_attention_chunkwise_gb300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def weights(Dd, L, seed):
    g = torch.Generator().manual_seed(seed)
    W1 = torch.randn((Dd, 2 * L), generator=g) / math.sqrt(Dd)
    W2 = torch.randn((2 * L, L), generator=g) / math.sqrt(2 * L)
    b = 0.54 + 0.3 * torch.randn((L,), generator=g)
    return W1, W2, b


@pytest.mark.parametrize("B,H,T,Dd,L,dtype", [(2, 3, 100, 64, 7, torch.float32),
                                              (1, 4, 333, 128, 12, torch.bfloat16),
                                              (1, 2, 64, 256, 25, torch.bfloat16),
                                              (3, 1, 7, 1, 1, torch.float32),
                                              # tensor-core first layer: K blocks of 64, padded
                                              # hidden widths, ragged last tile, several tiles per CTA
                                              (1, 2, 777, 192, 16, torch.bfloat16),
                                              (2, 1, 300, 64, 8, torch.bfloat16),
                                              (1, 4, 8192, 128, 14, torch.bfloat16),
                                              (1, 1, 5000, 128, 24, torch.bfloat16),
                                              (1, 1, 513, 64, 32, torch.bfloat16)])
def test_lambda_mlp_matches_oracle(B, H, T, Dd, L, dtype):
    g = torch.Generator().manual_seed(Dd + L)
    d = torch.randn((B, H, T, Dd), generator=g).to(dtype)
    W1, W2, b = weights(Dd, L, seed=L)
    lam = binding.lambda_mlp(d.cuda(), W1.cuda(), W2.cuda(), b.cuda())
    torch.cuda.synchronize()
    ref = oracle.lambda_mlp(d, W1, W2, b)
    np.testing.assert_allclose(lam.double().cpu().numpy(), ref, rtol=2e-5, atol=2e-6)


def test_lambda_mlp_initialisation_gives_one():
    d = torch.randn((1, 2, 300, 64), device="cuda")
    W1 = torch.randn((64, 18), device="cuda")
    lam = binding.lambda_mlp(d, W1, torch.zeros((18, 9), device="cuda"),
                             torch.full((9,), 0.54, device="cuda"))
    torch.cuda.synchronize()
    assert torch.allclose(lam, torch.full_like(lam, 0.99916), atol=1e-5)


def test_lambda_mlp_feeds_the_forward():
    """lambda from the MLP on the keys, then the tensor-core forward: the
    result matches the oracle run on the oracle's own lambda."""
    cfg = W.small_fwd_config(1, 4, 2048, 128, 128, 64, torch.bfloat16, seed=21)
    x = W.make_fwd_inputs(cfg)
    W1, W2, b = weights(128, cfg.L, seed=5)
    xd = {n: t.cuda() for n, t in x.items()}
    lam = binding.lambda_mlp(xd["k"], W1.cuda(), W2.cuda(), b.cuda())
    out = binding.fwd(xd["q"], xd["k"], xd["v"], xd["g"], lam, chunk=64)
    torch.cuda.synchronize()
    lam_ref = oracle.lambda_mlp(x["k"], W1, W2, b)
    np.testing.assert_allclose(lam.double().cpu().numpy(), lam_ref, rtol=2e-5, atol=2e-6)
    ref = oracle.naive(x["q"], x["k"], x["v"], x["g"], lam_ref)
    assert_parity(out, ref, torch.bfloat16, "forward on MLP lambda")


def test_lambda_mlp_full_size_sampled_rows():
    B, H, T, Dd, L = 1, 16, 32768, 128, 16
    g = torch.Generator(device="cuda").manual_seed(7)
    d = torch.randn((B, H, T, Dd), generator=g, device="cuda").bfloat16()
    W1, W2, b = weights(Dd, L, seed=8)
    lam = binding.lambda_mlp(d, W1.cuda(), W2.cuda(), b.cuda())
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, 127, 128, 4095, 16384, 32766, 32767])
    for h in (0, 7, 15):
        ref = oracle.lambda_mlp(d[0, h, rows].cpu(), W1, W2, b)
        np.testing.assert_allclose(lam[0, h, rows].double().cpu().numpy(), ref, rtol=2e-5, atol=2e-6)


def test_lambda_mlp_at_the_32k_workload_sampled_rows():
    """d = k of the T=32768 workload (B=1, H=16, Dd=128, bf16, L=16) as bench.py
    times it; 2048 sampled rows against the oracle."""
    cfg = W.FWD_CONFIGS["bf16_T32768_slowdecay"]
    k = W.make_fwd_inputs(cfg)["k"]
    W1, W2, b = weights(128, cfg.L, seed=9)
    lam = binding.lambda_mlp(k.cuda(), W1.cuda(), W2.cuda(), b.cuda())
    torch.cuda.synchronize()
    rows = torch.randint(0, cfg.H * cfg.T, (2048,), generator=torch.Generator().manual_seed(3))
    flat = lam.reshape(-1, cfg.L).cpu()[rows]
    ref = oracle.lambda_mlp(k.reshape(-1, 128)[rows], W1, W2, b)
    np.testing.assert_allclose(flat.double().numpy(), ref, rtol=2e-5, atol=2e-6)


def _fused_case(B, H, T, d, seed, separate_d=False, out_dtype=torch.float32):
    cfg = W.small_fwd_config(B, H, T, d, d, 64, torch.bfloat16, seed=seed)
    x = W.make_fwd_inputs(cfg)
    L = cfg.L
    W1, W2, b = weights(d, L, seed=seed + 1)
    dd = x["k"].clone() if separate_d else x["k"]
    lam_ref = oracle.lambda_mlp(dd, W1, W2, b)
    ref = oracle.naive(x["q"], x["k"], x["v"], x["g"], lam_ref)
    xd = {n: t.cuda() for n, t in x.items()}
    d_dev = dd.cuda() if separate_d else xd["k"]
    out = binding.fwd_lambda_mlp(xd["q"], xd["k"], xd["v"], xd["g"], d_dev, W1.cuda(), W2.cuda(), b.cuda(),
                                 chunk=64, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out, ref


@pytest.mark.parametrize("B,H,T,d", [(1, 2, 384, 128), (2, 2, 2048, 128), (1, 3, 1088, 64),
                                     (2, 2, 256, 64), (1, 1, 64, 128), (1, 2, 4224, 128)])
def test_fwd_lambda_mlp_in_the_read_out(B, H, T, d):
    """d = k on the tensor-core shapes: lambda computed inside the read-out
    from the key tile (never written to memory), against the oracle's MLP
    followed by the oracle's double sum."""
    out, ref = _fused_case(B, H, T, d, seed=T + d)
    assert_parity(out, ref, torch.bfloat16, f"fused lambda MLP {(B, H, T, d)}")


def test_fwd_lambda_mlp_two_pass_path_agrees():
    """A separate d tensor (same values as k) takes the two-pass path; both
    paths match the oracle, and each other to rounding."""
    out_sep, ref = _fused_case(1, 2, 1024, 128, seed=9, separate_d=True)
    out_fused, _ = _fused_case(1, 2, 1024, 128, seed=9)
    assert_parity(out_sep, ref, torch.bfloat16, "two-pass lambda MLP")
    assert_parity(out_fused, ref, torch.bfloat16, "fused lambda MLP")
    assert float((out_sep - out_fused).abs().max()) <= 1e-2


def test_fwd_lambda_mlp_bf16_out_and_cuda_core_shapes():
    out, ref = _fused_case(1, 2, 640, 64, seed=3, out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    d = out.double().cpu().numpy() - ref
    assert np.linalg.norm(d) / np.linalg.norm(ref) <= 5e-3
    # dk = 32 has no tensor-core path: the MLP runs first, then the CUDA-core forward
    out, ref = _fused_case(1, 2, 256, 32, seed=4)
    assert_parity(out, ref, torch.bfloat16, "lambda MLP, CUDA-core forward")
