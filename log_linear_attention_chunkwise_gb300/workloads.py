"""Seeded synthetic workloads for log-linear attention.

This module draws inputs and nothing else: it holds none of the operator's
arithmetic, and both the CUDA path's callers and the oracle's callers take
their inputs from here.  Every tensor comes from a ``torch.Generator`` seeded
per workload, drawn in a fixed order, so a (recipe, seed) pair fixes every
value.

Distributions (the workloads the pages' operator is exercised on; page
"Adaptive memory decay for Log-Linear Attention" §LambdaMLPSoftplus fixes the
lambda centre: softplus(0.54) is about 1.0 and softplus keeps lambda >= 0):
  q ~ N(0,1)/sqrt(dk);  k ~ N(0,1) then L2-normalised per token (in fp32);
  v ~ N(0,1);  g = -softplus(N(g_mu, 1)) per (batch, head, token);
  lambda = softplus(N(0.54, 0.3)) per (batch, head, token, level).
q, k, v are drawn in fp32 and rounded to the storage dtype (bf16:
round-to-nearest-even); g and lambda stay fp32.
"""

from __future__ import annotations

import dataclasses
import math

import torch


def num_levels(T: int) -> int:
    """1 + bit_length(T-1): level 0 plus the Fenwick levels of [0, T-1)."""
    return 1 + max(T - 1, 0).bit_length()


@dataclasses.dataclass(frozen=True)
class FwdConfig:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    chunk: int
    dtype: torch.dtype
    seed: int
    g_mu: float = 0.0            # g = -softplus(N(g_mu, 1))
    lam_one_frac: float = 0.0    # fraction of (head, level) pairs with lambda == 1
    g_zero_head_frac: float = 0.0  # fraction of heads with g == 0 (stress only)

    @property
    def L(self) -> int:
        return num_levels(self.T)

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "FwdConfig":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    H: int
    dk: int
    dv: int
    Ls: int
    steps: int
    pos_lo: int
    pos_hi: int
    dtype: torch.dtype
    seed: int


# The five workloads: four chunked forwards and one decode run.
FWD_CONFIGS = {
    "fp32_T256": FwdConfig("fp32_T256", 1, 2, 256, 32, 32, 16, torch.float32, 0),
    "bf16_T2048": FwdConfig("bf16_T2048", 4, 8, 2048, 64, 64, 64, torch.bfloat16, 1),
    "bf16_T8192_lam1": FwdConfig("bf16_T8192_lam1", 2, 16, 8192, 128, 128, 64,
                                 torch.bfloat16, 2, lam_one_frac=0.5),
    "bf16_T32768_slowdecay": FwdConfig("bf16_T32768_slowdecay", 1, 16, 32768, 128, 128, 64,
                                       torch.bfloat16, 3, g_mu=-2.0),
}
DECODE_CONFIG = DecodeConfig("decode_b64_h16_d128", batch=64, H=16, dk=128, dv=128,
                             Ls=17, steps=256, pos_lo=1, pos_hi=65536,
                             dtype=torch.bfloat16, seed=4)


def _softplus(x: torch.Tensor) -> torch.Tensor:
    return torch.nn.functional.softplus(x)


def make_fwd_inputs(cfg: FwdConfig, device="cpu") -> dict:
    """q, k, v [B,H,T,d] in cfg.dtype; g [B,H,T] fp32; lam [B,H,T,L] fp32."""
    gen = torch.Generator(device="cpu").manual_seed(cfg.seed)
    B, H, T, dk, dv, L = cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, cfg.L
    f32 = torch.float32
    q = torch.randn((B, H, T, dk), generator=gen, dtype=f32) / math.sqrt(dk)
    k = torch.randn((B, H, T, dk), generator=gen, dtype=f32)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    v = torch.randn((B, H, T, dv), generator=gen, dtype=f32)
    g = -_softplus(torch.randn((B, H, T), generator=gen, dtype=f32) + cfg.g_mu)
    lam = _softplus(0.54 + 0.3 * torch.randn((B, H, T, L), generator=gen, dtype=f32))
    if cfg.lam_one_frac > 0.0:
        # one (head, level) mask shared across batch and tokens
        mask = torch.rand((H, L), generator=gen) < cfg.lam_one_frac
        lam = torch.where(mask[None, :, None, :], torch.ones((), dtype=f32), lam)
    if cfg.g_zero_head_frac > 0.0:
        heads = torch.rand((H,), generator=gen) < cfg.g_zero_head_frac
        g = torch.where(heads[None, :, None], torch.zeros((), dtype=f32), g)
    out = {
        "q": q.to(cfg.dtype), "k": k.to(cfg.dtype), "v": v.to(cfg.dtype),
        "g": g.contiguous(), "lam": lam.contiguous(),
    }
    if device != "cpu":
        out = {n: t.to(device) for n, t in out.items()}
    return out


def small_fwd_config(B=1, H=2, T=256, dk=32, dv=32, chunk=16, dtype=torch.float32,
                     seed=0, g_mu=0.0, lam_one_frac=0.0, g_zero_head_frac=0.0,
                     name="custom") -> FwdConfig:
    return FwdConfig(name, B, H, T, dk, dv, chunk, dtype, seed, g_mu, lam_one_frac,
                     g_zero_head_frac)


# Log-Linear Gated DeltaNet: no workload on the pages; the 2K shape of the
# chunked forward with a per-token beta = sigmoid(N(0,1)).
GDN_CONFIG = FwdConfig("gdn_bf16_T2048", 4, 8, 2048, 64, 64, 64, torch.bfloat16, 5)


def make_gdn_inputs(cfg: FwdConfig, device="cpu") -> dict:
    """The forward inputs of cfg plus beta [B,H,T] fp32 in (0,1), drawn from a
    generator of its own (seed + 7919) so q, k, v, g, lambda match make_fwd_inputs."""
    x = make_fwd_inputs(cfg, device)
    gen = torch.Generator(device="cpu").manual_seed(cfg.seed + 7919)
    beta = torch.sigmoid(torch.randn((cfg.B, cfg.H, cfg.T), generator=gen, dtype=torch.float32))
    x["beta"] = beta.to(device) if device != "cpu" else beta
    return x


def make_decode_positions(cfg: DecodeConfig) -> torch.Tensor:
    """Start positions pos0 [batch] ~ U[pos_lo, pos_hi] (int64)."""
    gen = torch.Generator(device="cpu").manual_seed(cfg.seed)
    return torch.randint(cfg.pos_lo, cfg.pos_hi + 1, (cfg.batch,), generator=gen,
                         dtype=torch.int64)


def make_decode_prefix(cfg: DecodeConfig, pos0: torch.Tensor, Tp: int, device="cpu",
                       heads=None, seqs=None) -> dict:
    """Prefix keys, values and gates for decode states: k, v [b,h,Tp,d] in
    cfg.dtype and g [b,h,Tp] fp32, with the forward workloads' distributions.
    Values are drawn per (sequence, head) from a generator seeded with
    (seed, sequence, head), so any subset of (sequence, head) pairs can be
    regenerated on its own; entries at or beyond pos0[seq] are zeroed."""
    seqs = list(range(cfg.batch)) if seqs is None else list(seqs)
    heads = list(range(cfg.H)) if heads is None else list(heads)
    k = torch.empty((len(seqs), len(heads), Tp, cfg.dk), dtype=cfg.dtype, device=device)
    v = torch.empty((len(seqs), len(heads), Tp, cfg.dv), dtype=cfg.dtype, device=device)
    g = torch.empty((len(seqs), len(heads), Tp), dtype=torch.float32, device=device)
    gen_dev = device if str(device).startswith("cuda") else "cpu"
    for bi, b in enumerate(seqs):
        n = int(pos0[b])
        for hi, h in enumerate(heads):
            gen = torch.Generator(device=gen_dev).manual_seed(
                (cfg.seed * 1_000_003 + b * 1009 + h) & 0x7FFFFFFFFFFFFFFF)
            kk = torch.randn((Tp, cfg.dk), generator=gen, device=gen_dev)
            kk = kk / kk.norm(dim=-1, keepdim=True).clamp_min(1e-12)
            vv = torch.randn((Tp, cfg.dv), generator=gen, device=gen_dev)
            gg = -_softplus(torch.randn((Tp,), generator=gen, device=gen_dev))
            kk[n:] = 0
            vv[n:] = 0
            gg[n:] = 0
            k[bi, hi] = kk.to(cfg.dtype)
            v[bi, hi] = vv.to(cfg.dtype)
            g[bi, hi] = gg
    return {"k": k, "v": v, "g": g}


def make_decode_steps(cfg: DecodeConfig, device="cpu") -> dict:
    """Per-step decode inputs: q, k [steps,batch,H,dk], v [steps,batch,H,dv] in
    cfg.dtype; g [steps,batch,H] fp32; lam [steps,batch,H,Ls+1] fp32."""
    gen = torch.Generator(device="cpu").manual_seed(cfg.seed + 7919)
    S, Bn, H, dk, dv = cfg.steps, cfg.batch, cfg.H, cfg.dk, cfg.dv
    f32 = torch.float32
    q = torch.randn((S, Bn, H, dk), generator=gen, dtype=f32) / math.sqrt(dk)
    k = torch.randn((S, Bn, H, dk), generator=gen, dtype=f32)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    v = torch.randn((S, Bn, H, dv), generator=gen, dtype=f32)
    g = -_softplus(torch.randn((S, Bn, H), generator=gen, dtype=f32))
    lam = _softplus(0.54 + 0.3 * torch.randn((S, Bn, H, cfg.Ls + 1), generator=gen,
                                             dtype=f32))
    out = {"q": q.to(cfg.dtype), "k": k.to(cfg.dtype), "v": v.to(cfg.dtype),
           "g": g, "lam": lam}
    if device != "cpu":
        out = {n: t.to(device) for n, t in out.items()}
    return out
