"""lla_fwd_host (the forward on host buffers, pipelined over (batch, head)
groups) gives exactly the device forward's results."""

import pytest
import torch

from log_linear_attention_chunkwise_gb300 import binding
from log_linear_attention_chunkwise_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def both(cfg, group, pin=True, out_dtype=torch.float32, reps=1):
    x = W.make_fwd_inputs(cfg)
    hx = {n: (t.pin_memory() if pin else t.contiguous()) for n, t in x.items()}
    xd = {n: t.cuda() for n, t in x.items()}
    ref = binding.fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["lam"], chunk=cfg.chunk,
                      out_dtype=out_dtype)
    need = binding.load().lla_fwd_host_workspace_bytes(
        cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, cfg.chunk, binding._dt(x["q"]),
        binding._dt(torch.empty(0, dtype=out_dtype)), group)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(reps):
        out = torch.empty((cfg.B, cfg.H, cfg.T, cfg.dv), dtype=out_dtype, pin_memory=pin)
        binding.fwd_host(hx["q"], hx["k"], hx["v"], hx["g"], hx["lam"], out=out, chunk=cfg.chunk,
                         group=group, workspace=ws)
        outs.append(out)
    torch.cuda.synchronize()
    return ref.cpu(), outs


@pytest.mark.parametrize("group", [0, 1, 2, 5, 64])
def test_fwd_host_equals_device_forward_tensor_cores(group):
    cfg = W.small_fwd_config(2, 3, 384, 128, 128, 64, torch.bfloat16, seed=31)
    ref, outs = both(cfg, group, reps=2)
    for out in outs:
        assert torch.equal(out, ref)


def test_fwd_host_cuda_core_path_and_bf16_out():
    ref, outs = both(W.FWD_CONFIGS["fp32_T256"], 1)
    assert torch.equal(outs[0], ref)
    cfg = W.small_fwd_config(1, 4, 256, 64, 64, 32, torch.bfloat16, seed=2)
    ref, outs = both(cfg, 3, out_dtype=torch.bfloat16)
    assert torch.equal(outs[0], ref)


def test_fwd_host_pageable_buffers():
    cfg = W.small_fwd_config(1, 2, 512, 128, 128, 64, torch.bfloat16, seed=4)
    ref, outs = both(cfg, 1, pin=False)
    assert torch.equal(outs[0], ref)
