"""GPU parity of lla_decode_step and lla_prefill_state against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from log_linear_attention_chunkwise_gb300 import binding
from log_linear_attention_chunkwise_gb300 import workloads as W
from parity import assert_parity, errors

pytestmark = pytest.mark.gpu


def true_state(S, d):
    S = S.double().cpu().numpy() if isinstance(S, torch.Tensor) else S
    d = d.double().cpu().numpy() if isinstance(d, torch.Tensor) else d
    return np.exp(d)[..., None, None] * S


def live_mask(pos, Ls):
    return np.array([[(int(p) >> i) & 1 for i in range(Ls)] for p in pos], bool)


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 64, 64), (torch.float32, 32, 16),
                                         (torch.bfloat16, 128, 128), (torch.float32, 16, 128)])
def test_replay_from_empty_state_matches_double_sum(dtype, dk, dv):
    B, H, T = 2, 3, 300
    cfg = W.small_fwd_config(B, H, T, dk, dv, 16, dtype, seed=dk + dv)
    x = W.make_fwd_inputs(cfg)
    ref = oracle.naive(x["q"], x["k"], x["v"], x["g"], x["lam"])
    Ls = T.bit_length()
    L = cfg.L
    xd = {n: t.cuda() for n, t in x.items()}
    S = torch.zeros((B, H, Ls, dk, dv), device="cuda")
    D = torch.zeros((B, H, Ls), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for t in range(T):
        lam_t = torch.zeros((B, H, Ls + 1), device="cuda")
        lam_t[..., :L] = xd["lam"][:, :, t]
        pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        outs.append(binding.decode_step(S, D, xd["q"][:, :, t].contiguous(),
                                        xd["k"][:, :, t].contiguous(),
                                        xd["v"][:, :, t].contiguous(),
                                        xd["g"][:, :, t].contiguous(), lam_t, pos,
                                        device_error=err))
    out = torch.stack(outs, dim=2)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_parity(out, ref, dtype, "decode replay")
    # the final state is the bucket state of [0, T)
    S_cf, _ = oracle.state_closed_form(x["k"], x["v"], x["g"], np.full(B, T), Ls)
    live = live_mask([T], Ls)[0]
    max_abs, rel_fro, _ = errors(true_state(S, D)[:, :, live], S_cf[:, :, live])
    assert rel_fro <= (5e-3 if dtype == torch.bfloat16 else 1e-4), rel_fro


@pytest.mark.parametrize("T,dtype,d", [(1000, torch.bfloat16, 64), (777, torch.float32, 32),
                                       (4096, torch.bfloat16, 128), (1, torch.float32, 16),
                                       (0, torch.bfloat16, 64)])
def test_prefill_state_matches_closed_form(T, dtype, d):
    B, H = 2, 2
    Ls = max(T.bit_length(), 1) + 1
    cfg = W.small_fwd_config(B, H, max(T, 1), d, d, 1, dtype, seed=T)
    x = W.make_fwd_inputs(cfg)
    k, v, g = (x[n][:, :, :T].contiguous() for n in ("k", "v", "g"))
    S, D = binding.prefill_state(k.cuda(), v.cuda(), g.cuda(), Ls)
    torch.cuda.synchronize()
    assert torch.count_nonzero(D) == 0
    S_cf, _ = oracle.state_closed_form(k, v, g, np.full(B, T), Ls)
    max_abs, rel_fro, _ = errors(S, S_cf)
    if T > 0:
        assert rel_fro <= (1e-3 if dtype == torch.bfloat16 else 1e-5), rel_fro
    dead = ~live_mask([T], Ls)[0]
    assert torch.count_nonzero(S[:, :, torch.from_numpy(dead)]) == 0


def test_prefill_then_decode_continues_the_sequence():
    B, H, T, d = 2, 2, 700, 64
    cfg = W.small_fwd_config(B, H, T, d, d, 16, torch.bfloat16, seed=77)
    x = W.make_fwd_inputs(cfg)
    xd = {n: t.cuda() for n, t in x.items()}
    p0 = 613
    Ls = T.bit_length()
    S, D = binding.prefill_state(xd["k"][:, :, :p0].contiguous(), xd["v"][:, :, :p0].contiguous(),
                                 xd["g"][:, :, :p0].contiguous(), Ls)
    rows = list(range(p0, T))
    outs = []
    for t in rows:
        lam_t = torch.zeros((B, H, Ls + 1), device="cuda")
        lam_t[..., :cfg.L] = xd["lam"][:, :, t]
        pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        outs.append(binding.decode_step(S, D, xd["q"][:, :, t].contiguous(),
                                        xd["k"][:, :, t].contiguous(),
                                        xd["v"][:, :, t].contiguous(),
                                        xd["g"][:, :, t].contiguous(), lam_t, pos))
    out = torch.stack(outs, dim=2).cpu()
    for b in range(B):
        for h in range(H):
            ref = oracle.naive_rows(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["g"][b, h],
                                    x["lam"][b, h], rows)
            assert_parity(out[b, h], ref, torch.bfloat16, f"continue {(b, h)}")


def test_position_without_room_sets_device_error():
    B, H, d, Ls = 3, 2, 64, 4
    S = torch.randn((B, H, Ls, d, d), device="cuda")
    D = torch.zeros((B, H, Ls), device="cuda")
    S0 = S.clone()
    q = torch.randn((B, H, d), device="cuda").bfloat16()
    g = -torch.rand((B, H), device="cuda")
    lam = torch.ones((B, H, Ls + 1), device="cuda")
    pos = torch.tensor([3, 15, 5], dtype=torch.int64, device="cuda")  # 15+1 needs 5 slots
    out = torch.full((B, H, d), 7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.decode_step(S, D, q, q, q, g, lam, pos, out=out, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 2  # 1 + index of the offending sequence
    assert torch.equal(S[1], S0[1]) and torch.all(out[1] == 7.0)
    assert not torch.all(out[0] == 7.0)


def test_decode_workload_sampled_pairs():
    """64 sequences at positions in [1, 65536], states built from their
    prefixes with lla_prefill_state, then 256 decode steps; sampled
    (sequence, head) pairs follow the oracle from its own closed-form state."""
    cfg = W.DECODE_CONFIG
    pos0 = W.make_decode_positions(cfg)
    steps = W.make_decode_steps(cfg, device="cuda")
    Bn, H, dk, dv, Ls = cfg.batch, cfg.H, cfg.dk, cfg.dv, cfg.Ls
    S = torch.empty((Bn, H, Ls, dk, dv), device="cuda")
    D = torch.empty((Bn, H, Ls), device="cuda")
    for b in range(Bn):
        n = int(pos0[b])
        pre = W.make_decode_prefix(cfg, pos0, n, device="cuda", seqs=[b])
        binding.prefill_state(pre["k"], pre["v"], pre["g"], Ls, state=S[b:b + 1], logdecay=D[b:b + 1])
        del pre
    pos_dev = pos0.cuda()
    outs = []
    for s in range(cfg.steps):
        outs.append(binding.decode_step(S, D, steps["q"][s], steps["k"][s], steps["v"][s],
                                        steps["g"][s], steps["lam"][s], pos_dev + s))
    out = torch.stack(outs).cpu()  # [steps, B, H, dv]
    S_end = S.cpu()
    D_end = D.cpu()
    torch.cuda.synchronize()
    # 16 (sequence, head) pairs: the longest and shortest prefixes, then a
    # seeded draw over the other sequences, every head at least once
    rng = np.random.default_rng(44)
    seqs = [int(np.argmax(pos0)), int(np.argmin(pos0))]
    seqs += [int(b) for b in rng.permutation(Bn) if int(b) not in seqs][:14]
    pairs = [(b, i % H) for i, b in enumerate(seqs)]
    assert len(set(pairs)) == 16 and {h for _, h in pairs} == set(range(H))
    for (b, h) in pairs:
        n = int(pos0[b])
        pre = W.make_decode_prefix(cfg, pos0, n, device="cuda", seqs=[b], heads=[h])
        So, Do = oracle.state_closed_form(pre["k"].cpu(), pre["v"].cpu(), pre["g"].cpu(), [n], Ls)
        ref = []
        for s in range(cfg.steps):
            ref.append(oracle.decode_step(So, Do, steps["q"][s, b:b + 1, h:h + 1].cpu(),
                                          steps["k"][s, b:b + 1, h:h + 1].cpu(),
                                          steps["v"][s, b:b + 1, h:h + 1].cpu(),
                                          steps["g"][s, b:b + 1, h:h + 1].cpu(),
                                          steps["lam"][s, b:b + 1, h:h + 1].cpu(), [n + s])[0, 0])
        assert_parity(out[:, b, h], np.stack(ref), torch.bfloat16, f"decode pair {(b, h)}")
        live = live_mask([n + cfg.steps], Ls)[0]
        _, rel_fro, _ = errors(true_state(S_end[b, h], D_end[b, h])[live],
                               true_state(So[0, 0], Do[0, 0])[live])
        assert rel_fro <= 5e-3, rel_fro


@pytest.mark.parametrize("T", [100, 300, 2944, 16384])
def test_prefill_state_tensor_core_buckets(T):
    """bf16, dk = dv = 128: the tensor-core bucket path, with buckets shorter
    than a 128-token tile, buckets that start off a tile boundary and a
    multi-CTA bucket."""
    B, H, d = 1, 2, 128
    Ls = T.bit_length()
    cfg = W.small_fwd_config(B, H, T, d, d, 1, torch.bfloat16, seed=T + 1)
    x = W.make_fwd_inputs(cfg)
    S, D = binding.prefill_state(x["k"].cuda(), x["v"].cuda(), x["g"].cuda(), Ls)
    torch.cuda.synchronize()
    pos = np.full(B, T)
    S_cf, _ = oracle.state_closed_form(x["k"], x["v"], x["g"], pos, Ls)
    live = live_mask(pos, Ls)[0]
    Sn = S.cpu().double().numpy()
    max_abs, rel_fro, _ = errors(Sn[:, :, live], S_cf[:, :, live])
    assert rel_fro <= 1e-3, rel_fro
    if (~live).any():
        assert np.abs(Sn[:, :, ~live]).max() == 0.0


def test_prefill_state_at_the_32k_workload():
    """k, v, g of the T=32768 workload (B=1, H=16, d=128, bf16) as bench.py times
    it: the state of two heads against the closed form."""
    cfg = W.FWD_CONFIGS["bf16_T32768_slowdecay"]
    x = W.make_fwd_inputs(cfg)
    Ls = cfg.T.bit_length()
    S, D = binding.prefill_state(x["k"].cuda(), x["v"].cuda(), x["g"].cuda(), Ls)
    torch.cuda.synchronize()
    assert float(D.abs().max()) == 0.0
    for h in (3, 15):
        sl = {n: t[:, h:h + 1] for n, t in x.items()}
        S_cf, _ = oracle.state_closed_form(sl["k"], sl["v"], sl["g"], np.array([cfg.T]), Ls)
        live = live_mask(np.array([cfg.T]), Ls)[0]
        Sn = S[:, h:h + 1].cpu().double().numpy()
        max_abs, rel_fro, _ = errors(Sn[:, :, live], S_cf[:, :, live])
        assert rel_fro <= 1e-3, (h, rel_fro)
