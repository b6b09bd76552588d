"""lla_fwd_noalloc: the forward for callers that cannot allocate device memory.

It takes no workspace; its scratch is a fixed array inside the library.  This
file is collected last so that a failure here leaves every other test already
run.  It checks, through the C ABI, that two calls in a row give what the
workspace entry point gives, on the tensor-core path and the CUDA-core path,
and that a call needing more scratch than the array holds is refused.
"""

import ctypes

import pytest
import torch

from log_linear_attention_chunkwise_gb300 import binding
from log_linear_attention_chunkwise_gb300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def noalloc_fwd(lib, x, chunk, out):
    B, H, T, dk = x["q"].shape
    dv = x["v"].shape[-1]
    in_dt = binding.LLA_BF16 if x["q"].dtype == torch.bfloat16 else binding.LLA_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.lla_fwd_noalloc(_p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["g"]), _p(x["lam"]),
                               _p(out), B, H, T, dk, dv, chunk, in_dt, binding.LLA_F32, None, stream)


@pytest.mark.parametrize("B,H,T,d,chunk,dtype", [
    (1, 4, 2048, 128, 64, torch.bfloat16),   # tensor-core kernels
    (2, 2, 512, 64, 64, torch.bfloat16),     # CUDA-core kernels
    (1, 2, 256, 32, 16, torch.float32),
])
def test_noalloc_matches_workspace_entry_point_twice(B, H, T, d, chunk, dtype):
    lib = binding.load()
    cfg = W.small_fwd_config(B, H, T, d, d, chunk, dtype, seed=T + d)
    x = {n: t.cuda() for n, t in W.make_fwd_inputs(cfg).items()}
    ref = binding.fwd(x["q"], x["k"], x["v"], x["g"], x["lam"], chunk=chunk)
    torch.cuda.synchronize()
    assert lib.lla_fwd_workspace_bytes(B, H, T, d, d, chunk, 1 if dtype == torch.bfloat16 else 0) \
        <= lib.lla_fwd_noalloc_max_scratch_bytes()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert noalloc_fwd(lib, x, chunk, out) == 0
        torch.cuda.synchronize()
        assert_parity(out, ref.double().cpu().numpy(), dtype, f"no-alloc call {call}")


def test_noalloc_refuses_more_than_its_scratch():
    lib = binding.load()
    limit = lib.lla_fwd_noalloc_max_scratch_bytes()
    assert limit == 64 << 20
    # 16 heads x 32768 tokens at d = 128 needs far more than 64 MiB
    B, H, T, d = 1, 16, 32768, 128
    assert lib.lla_fwd_workspace_bytes(B, H, T, d, d, 64, 1) > limit
    # real, aligned device buffers, so only the scratch size can be refused
    q = torch.zeros((B, H, T, d), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((B, H, T), dtype=torch.float32, device="cuda")
    lam = torch.zeros((B, H, T, lib.lla_num_levels(T)), dtype=torch.float32, device="cuda")
    out = torch.full((B, H, T, d), 7.0, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.lla_fwd_noalloc(_p(q), _p(q), _p(q), _p(g), _p(lam), _p(out), B, H, T, d, d, 64, 1, 0,
                             None, stream)
    assert rc == 3  # LLA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # nothing was enqueued
