"""GPU parity of lla_fwd against the fp64 oracle (through the C ABI).

Every case compares every output element.  The full-size workloads (and a
zero-gate stress variant of the T=32768 one) are compared head by head with
the oracle's Fenwick recurrence, plus sampled rows against the double sum
(an independent form of the same operator), and the T=32768 workload checks
chunk-size invariance over the whole tensor.
"""

import numpy as np
import pytest
import torch

import oracle
from log_linear_attention_chunkwise_gb300 import binding
from log_linear_attention_chunkwise_gb300 import workloads as W
from parity import assert_parity, errors

pytestmark = pytest.mark.gpu


def to_dev(x):
    return {n: t.to("cuda") for n, t in x.items()}


def gpu_fwd(xd, chunk, out_dtype=torch.float32):
    out = binding.fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["lam"], chunk=chunk,
                      out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out


def oracle_full(x):
    return oracle.naive(x["q"], x["k"], x["v"], x["g"], x["lam"])


SMALL = [
    # B, H, T, dk, dv, chunk, dtype, extra
    (1, 2, 256, 32, 32, 16, torch.float32, {}),
    (1, 1, 48, 16, 16, 16, torch.float32, {}),
    (2, 1, 128, 64, 64, 128, torch.float32, {}),
    (1, 2, 512, 64, 32, 32, torch.float32, {}),
    (1, 1, 192, 128, 128, 64, torch.float32, {}),
    (1, 2, 384, 128, 128, 64, torch.bfloat16, {}),
    (2, 2, 320, 64, 64, 64, torch.bfloat16, {}),
    (1, 1, 64, 64, 64, 64, torch.bfloat16, {}),
    (1, 1, 1024, 128, 128, 128, torch.bfloat16, {}),
    (1, 2, 256, 16, 16, 16, torch.bfloat16, {}),
    (1, 2, 640, 128, 64, 32, torch.bfloat16, {}),
    (1, 4, 1024, 64, 64, 64, torch.bfloat16, dict(g_zero_head_frac=0.5)),
    (1, 2, 1152, 128, 128, 64, torch.bfloat16, dict(g_mu=-6.0, lam_one_frac=0.5)),
    (1, 2, 320, 128, 128, 64, torch.bfloat16, {}),
    (2, 3, 64, 128, 128, 64, torch.bfloat16, {}),
    (1, 2, 2112, 128, 128, 64, torch.bfloat16, dict(g_zero_head_frac=0.5)),
    (1, 1, 4096, 128, 128, 32, torch.bfloat16, dict(g_mu=-3.0)),
]


@pytest.mark.parametrize("B,H,T,dk,dv,chunk,dtype,extra", SMALL)
def test_small_shapes_every_element(B, H, T, dk, dv, chunk, dtype, extra):
    cfg = W.small_fwd_config(B, H, T, dk, dv, chunk, dtype, seed=T + dk, **extra)
    x = W.make_fwd_inputs(cfg)
    out = gpu_fwd(to_dev(x), chunk)
    assert_parity(out, oracle_full(x), dtype, f"{cfg}", stress=cfg.g_zero_head_frac > 0)


def test_fp32_workload_full():
    cfg = W.FWD_CONFIGS["fp32_T256"]
    x = W.make_fwd_inputs(cfg)
    assert_parity(gpu_fwd(to_dev(x), cfg.chunk), oracle_full(x), cfg.dtype, cfg.name)


def test_bf16_T2048_workload_full():
    cfg = W.FWD_CONFIGS["bf16_T2048"]
    x = W.make_fwd_inputs(cfg)
    assert_parity(gpu_fwd(to_dev(x), cfg.chunk), oracle_full(x), cfg.dtype, cfg.name)


def test_bf16_T2048_stress_no_decay_heads():
    """g == 0 on a quarter of the heads: the multi-chunk Fenwick nodes then
    carry most of the output, so a wrong cross-chunk decay cannot hide."""
    cfg = W.FWD_CONFIGS["bf16_T2048"].with_(B=1, g_zero_head_frac=0.25, seed=11)
    x = W.make_fwd_inputs(cfg)
    assert_parity(gpu_fwd(to_dev(x), cfg.chunk), oracle_full(x), cfg.dtype, "stress", stress=True)


def test_bf16_output_dtype():
    cfg = W.FWD_CONFIGS["bf16_T2048"].with_(B=1, H=4)
    x = W.make_fwd_inputs(cfg)
    ref = oracle_full(x)
    out = gpu_fwd(to_dev(x), cfg.chunk, out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    max_abs, rel_fro, _ = errors(out, ref)
    # bf16 rounding of the result adds up to 2^-9 relative per element
    assert rel_fro <= 5e-3
    assert np.all(np.abs(out.double().cpu().numpy() - ref) <= 2e-2 + 2.0 ** -8 * np.abs(ref))


def sampled_rows(T, chunk, n_random, seed):
    rng = np.random.default_rng(seed)
    rows = {0, 1, chunk - 1, chunk, chunk + 1, 2 * chunk - 1, T // 2, T // 2 - 1, T - 2, T - 1}
    rows |= {int(r) for r in rng.integers(0, T, n_random)}
    rows |= {int(c) * chunk - 1 for c in rng.integers(1, T // chunk + 1, 8)}
    return sorted(r for r in rows if 0 <= r < T)


def check_full_size(cfg, pairs_rows, n_rows):
    """Every element of every head against the Fenwick recurrence (each head
    judged on its own, so one bad head cannot hide in the tensor's norm),
    then sampled rows of a few heads against the double sum."""
    x = W.make_fwd_inputs(cfg)
    xd = to_dev(x)
    out = gpu_fwd(xd, cfg.chunk)
    out_cpu = out.double().cpu().numpy()
    stress = cfg.g_zero_head_frac > 0
    ref = oracle.fenwick(x["q"], x["k"], x["v"], x["g"], x["lam"])
    for b in range(cfg.B):
        for h in range(cfg.H):
            assert_parity(out_cpu[b, h], ref[b, h], cfg.dtype, f"{cfg.name} head {(b, h)}",
                          stress=stress)
    assert_parity(out_cpu, ref, cfg.dtype, f"{cfg.name} all heads", stress=stress)
    del ref
    for i, (b, h) in enumerate(pairs_rows):
        rows = sampled_rows(cfg.T, cfg.chunk, n_rows, seed=100 + i)
        ref = oracle.naive_rows(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["g"][b, h],
                                x["lam"][b, h], rows)
        assert_parity(out_cpu[b, h, rows], ref, cfg.dtype, f"{cfg.name} rows of {(b, h)}",
                      stress=stress)
    return xd, out


def test_bf16_T8192_lambda_one_workload():
    cfg = W.FWD_CONFIGS["bf16_T8192_lam1"]
    check_full_size(cfg, pairs_rows=[(0, 0), (0, 7), (1, 15)], n_rows=24)


def test_bf16_T32768_workload_and_chunk_invariance():
    cfg = W.FWD_CONFIGS["bf16_T32768_slowdecay"]
    xd, out = check_full_size(cfg, pairs_rows=[(0, 0), (0, 9), (0, 15)], n_rows=24)
    # the operator does not depend on the chunk size: compare whole tensors
    for chunk in (32, 128):
        other = gpu_fwd(xd, chunk)
        max_abs, rel_fro, _ = errors(other, out.double().cpu().numpy())
        assert max_abs <= 2e-2 and rel_fro <= 5e-3, (chunk, max_abs, rel_fro)
    del xd, out
    torch.cuda.empty_cache()


def test_bf16_T32768_stress_no_decay_heads():
    """The T=32768 workload with g == 0 on 5 of its 16 heads (seed 20): there
    the nodes that span 4096-token segments (64, 96, 128, ... tiles), which
    the segment fix-up chains, carry most of the output, so a wrong chain
    over several segments cannot hide behind decay."""
    cfg = W.FWD_CONFIGS["bf16_T32768_slowdecay"].with_(g_zero_head_frac=0.25, seed=20,
                                                       name="bf16_T32768_stress")
    x = W.make_fwd_inputs(cfg)
    zero_heads = (x["g"][0].abs().sum(-1) == 0).nonzero().flatten().tolist()
    assert len(zero_heads) >= 2, zero_heads
    del x
    xd, out = check_full_size(cfg, pairs_rows=[(0, zero_heads[0]), (0, zero_heads[-1])], n_rows=16)
    del xd, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,d", [(4224, 64), (12288, 64), (12288, 128)])
def test_multi_segment_fixup_chain_stress(T, d):
    """Zero-gate heads at lengths with one, two or three full 32-tile
    segments, so the fix-up chain of segment totals (Node_32, Node_64, ...)
    carries most of the output, for both tensor-core widths."""
    cfg = W.small_fwd_config(1, 2, T, d, d, 64, torch.bfloat16, seed=T + 3 * d + 1, g_zero_head_frac=0.5)
    assert (W.make_fwd_inputs(cfg)["g"][0].abs().sum(-1) == 0).any()  # a head without decay
    check_full_size(cfg, pairs_rows=[], n_rows=0)


def test_bf16_T8192_stress_reduced():
    cfg = W.FWD_CONFIGS["bf16_T8192_lam1"].with_(B=1, H=4, g_zero_head_frac=0.5, seed=12)
    check_full_size(cfg, pairs_rows=[], n_rows=0)


@pytest.mark.parametrize("d", [64, 128])
def test_degenerate_inputs(d):
    cfg = W.small_fwd_config(1, 2, 512, d, d, 64, torch.bfloat16, seed=5)
    x = W.make_fwd_inputs(cfg)
    # lambda == 0 everywhere: exactly zero output
    xz = dict(x, lam=torch.zeros_like(x["lam"]))
    out = gpu_fwd(to_dev(xz), 64)
    assert torch.count_nonzero(out) == 0
    # a huge decay: only the diagonal survives (exp underflows to 0 on both sides)
    xd = dict(x, g=torch.full_like(x["g"], -1e4))
    assert_parity(gpu_fwd(to_dev(xd), 64), oracle_full(xd), cfg.dtype, "huge decay")
    # no decay at all
    x0 = dict(x, g=torch.zeros_like(x["g"]))
    assert_parity(gpu_fwd(to_dev(x0), 64), oracle_full(x0), cfg.dtype, "no decay", stress=True)


def test_empty_and_single_chunk():
    q = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device="cuda")
    lam = torch.empty((1, 2, 0, 1), dtype=torch.float32, device="cuda")
    g = torch.empty((1, 2, 0), dtype=torch.float32, device="cuda")
    out = binding.fwd(q, q, q, g, lam, chunk=64)
    assert out.shape == (1, 2, 0, 64)
    cfg = W.small_fwd_config(1, 1, 16, 16, 16, 16, torch.float32, seed=3)
    x = W.make_fwd_inputs(cfg)
    assert_parity(gpu_fwd(to_dev(x), 16), oracle_full(x), cfg.dtype, "T=16")


def test_deterministic():
    cfg = W.FWD_CONFIGS["bf16_T2048"].with_(B=1, H=2)
    xd = to_dev(W.make_fwd_inputs(cfg))
    a = gpu_fwd(xd, 64)
    b = gpu_fwd(xd, 64)
    assert torch.equal(a, b)


def test_workspace_too_small_is_rejected():
    cfg = W.FWD_CONFIGS["bf16_T2048"].with_(B=1, H=1)
    xd = to_dev(W.make_fwd_inputs(cfg))
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.LLAError) as e:
        binding.fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["lam"], chunk=64, workspace=ws)
    assert e.value.code == 3
