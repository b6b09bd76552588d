"""GPU parity of Log-Linear Gated DeltaNet (lla_gdn_fwd, lla_gdn_decode_step)
against the fp64 oracle's pair form and decode step.

The kernels compute in fp32 for both input dtypes and the oracle reads the
same rounded inputs, so the fp32 bound applies to every output:
||gpu - oracle||_F / ||oracle||_F <= 1e-4 and max |gpu - oracle| <= 1e-4 max |oracle|.
"""

import numpy as np
import pytest
import torch

import oracle
from log_linear_attention_chunkwise_gb300 import binding
from log_linear_attention_chunkwise_gb300 import workloads as W
from parity import errors

pytestmark = pytest.mark.gpu

REL = 1e-4


def check(got, ref, what):
    max_abs, rel_fro, ref_max = errors(got, ref)
    assert rel_fro <= REL and max_abs <= REL * max(ref_max, 1e-30), (
        f"{what}: max_abs={max_abs:.3e} (ref max {ref_max:.3e}) rel_fro={rel_fro:.3e}")


def run_fwd(cfg, state_Ls=0):
    x = W.make_gdn_inputs(cfg)
    d = {n: t.cuda() for n, t in x.items()}
    res = binding.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], state_Ls=state_Ls)
    torch.cuda.synchronize()
    return x, res


@pytest.mark.parametrize("B,H,T,dk,dv,dtype", [
    (1, 2, 64, 16, 16, torch.float32),      # one full chunk
    (2, 1, 100, 32, 64, torch.float32),     # a ragged second chunk
    (1, 1, 1, 64, 32, torch.float32),       # one token: only the diagonal
    (1, 1, 65, 64, 16, torch.float32),      # one token past the first chunk
    (1, 2, 333, 64, 64, torch.bfloat16),
    (1, 1, 256, 128, 128, torch.bfloat16),
    (1, 1, 512, 128, 16, torch.float32),
    (1, 1, 1024, 16, 128, torch.bfloat16),  # 16 chunks: four chunk levels live at once
    (2, 1, 1000, 32, 32, torch.float32),
])
def test_gdn_fwd_matches_oracle(B, H, T, dk, dv, dtype):
    cfg = W.small_fwd_config(B, H, T, dk, dv, 16, dtype, seed=T + dv)
    x, out = run_fwd(cfg)
    ref = oracle.gdn_naive(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"])
    check(out, ref, f"T{T} dk{dk} dv{dv}")


def test_gdn_fwd_lambda_one_is_gated_deltanet():
    cfg = W.small_fwd_config(1, 2, 200, 32, 32, 16, torch.float32, seed=8)
    x = W.make_gdn_inputs(cfg)
    x["lam"] = torch.ones_like(x["lam"])
    d = {n: t.cuda() for n, t in x.items()}
    out = binding.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"])
    torch.cuda.synchronize()
    check(out, oracle.gdn_base(x["q"], x["k"], x["v"], x["g"], x["beta"]), "lambda=1")


@pytest.mark.parametrize("T,dk,dv", [(45, 32, 32), (128, 32, 32), (200, 64, 32), (448, 16, 64), (513, 32, 16)])
def test_gdn_final_state_matches_the_oracle(T, dk, dv):
    """The state after the sequence (decode layout, every slot compared, the
    dead ones zero) against the oracle's decode steps from the empty state:
    chunk-level slots from the scan, the low-bit slots of a ragged end from
    the last chunk's buckets."""
    B, H = 1, 2
    cfg = W.small_fwd_config(B, H, T, dk, dv, 16, torch.float32, seed=T + 5)
    x = W.make_gdn_inputs(cfg)
    Ls = T.bit_length() + 1
    d = {n: t.cuda() for n, t in x.items()}
    out, S = binding.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], state_Ls=Ls)
    torch.cuda.synchronize()
    check(out, oracle.gdn_naive(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"]), f"T{T} out")
    S_ref = np.zeros((B, H, Ls, dk, dv))
    q, k, v, g, beta, lam = (x[n].double().numpy() for n in ("q", "k", "v", "g", "beta", "lam"))
    for t in range(T):
        lam_t = np.zeros((B, H, Ls + 1))
        lam_t[..., :lam.shape[-1]] = lam[:, :, t]
        oracle.gdn_decode_step(S_ref, q[:, :, t], k[:, :, t], v[:, :, t], g[:, :, t], beta[:, :, t], lam_t,
                               np.full((B,), t))
    S = S.cpu().double().numpy()
    live = [i for i in range(Ls) if (T >> i) & 1]
    # the live slots as one state: a deep slot can decay below fp32's range
    # (1e-70 in fp64 at T = 448), so its error is measured against the state
    check(S[:, :, live], S_ref[:, :, live], f"T{T} live slots {live}")
    for i in range(Ls):
        if i not in live:
            assert not S[:, :, i].any(), f"T{T} dead slot {i} not zero"


def test_gdn_workload_sampled_heads():
    """The 2K workload (B=4, H=8, T=2048, d=64, bf16); the oracle checks two
    (batch, head) pairs in full."""
    cfg = W.GDN_CONFIG
    x, out = run_fwd(cfg)
    for b, h in ((0, 0), (3, 5)):
        sl = {n: t[b:b + 1, h:h + 1] for n, t in x.items()}
        ref = oracle.gdn_naive(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], sl["lam"])
        check(out[b:b + 1, h:h + 1], ref, f"b{b} h{h}")


def test_gdn_prefill_then_decode_continues_the_sequence():
    """Forward over the first T0 tokens with the final state, then decode steps
    for the rest: every output equals the pair form over the whole sequence."""
    B, H, T, T0, d = 2, 2, 80, 45, 32
    cfg = W.small_fwd_config(B, H, T, d, d, 16, torch.float32, seed=3)
    x = W.make_gdn_inputs(cfg)
    ref = oracle.gdn_naive(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"])
    Ls = T.bit_length()
    d_ = {n: t.cuda() for n, t in x.items()}
    L0 = binding.load().lla_num_levels(T0)
    pre = {n: t[:, :, :T0].contiguous() for n, t in d_.items()}
    pre["lam"] = pre["lam"][..., :L0].contiguous()
    out0, S = binding.gdn_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], pre["lam"],
                              state_Ls=Ls)
    outs = [out0]
    for t in range(T0, T):
        lam_t = torch.zeros((B, H, Ls + 1), device="cuda")
        lam_t[..., :x["lam"].shape[-1]] = d_["lam"][:, :, t]
        pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        o = binding.gdn_decode_step(S, d_["q"][:, :, t].contiguous(), d_["k"][:, :, t].contiguous(),
                                    d_["v"][:, :, t].contiguous(), d_["g"][:, :, t].contiguous(),
                                    d_["beta"][:, :, t].contiguous(), lam_t, pos)
        outs.append(o[:, :, None])
    torch.cuda.synchronize()
    check(torch.cat(outs, dim=2), ref, "prefill + decode")


def test_gdn_decode_step_on_a_random_state():
    B, H, dk, dv, Ls = 3, 2, 64, 32, 17
    rng = np.random.default_rng(11)
    S = rng.standard_normal((B, H, Ls, dk, dv)) * 0.1
    pos = np.array([5, 1023, 65534])
    q = rng.standard_normal((B, H, dk)) / 8
    k = rng.standard_normal((B, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, H))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, H))))
    lam = np.log1p(np.exp(0.54 + 0.3 * rng.standard_normal((B, H, Ls + 1))))
    t32 = lambda a: torch.tensor(a, dtype=torch.float32, device="cuda").contiguous()
    Sg = t32(S)
    out = binding.gdn_decode_step(Sg, t32(q), t32(k), t32(v), t32(g), t32(beta), t32(lam),
                                  torch.tensor(pos, device="cuda"))
    torch.cuda.synchronize()
    S_ref = S.copy()
    ref = oracle.gdn_decode_step(S_ref, q, k, v, g, beta, lam, pos)
    check(out, ref, "decode out")
    Sg = Sg.cpu().double().numpy()
    for b, t in enumerate(pos.tolist()):
        m = ((t + 1) & -(t + 1)).bit_length() - 1
        keep = [i for i in range(Ls) if (t >> i) & 1 and i >= m] + [m]  # live slots that stay, and the new one
        check(Sg[b][:, keep], S_ref[b][:, keep], f"state b{b}")


def test_gdn_decode_reports_a_state_without_room():
    B, H, d, Ls = 2, 1, 16, 4
    S = torch.zeros((B, H, Ls, d, d), device="cuda")
    z = torch.zeros((B, H, d), device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    pos = torch.tensor([3, 15], dtype=torch.int64, device="cuda")  # bit_length(16) = 5 > 4
    binding.gdn_decode_step(S, z, z, z, torch.zeros((B, H), device="cuda"),
                            torch.zeros((B, H), device="cuda"), torch.zeros((B, H, Ls + 1), device="cuda"),
                            pos, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 2


def test_gdn_empty_is_a_noop():
    z = torch.empty((0, 2, 64, 32), device="cuda")
    out = binding.gdn_fwd(z, z, z, torch.empty((0, 2, 64), device="cuda"),
                          torch.empty((0, 2, 64), device="cuda"),
                          torch.empty((0, 2, 64, 7), device="cuda"))
    assert out.numel() == 0
