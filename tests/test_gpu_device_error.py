"""Device-detected failures reach the caller.

The tensor-core kernels bound every wait on a shared-memory barrier; a wait
that runs out records an lla_device_error code in the caller's device_error
word and the kernel runs to its end.  The library's test hook withholds the
first product of each tile (nothing is issued for it, so no copy or product
is left in flight) and bounds the waits at a few thousand polls, so the
waits on that product run out on purpose, in a small case, without any
fault.  The word must then read LLA_DEVERR_SYNC_TIMEOUT through
lla_device_error_check (status LLA_ERR_DEVICE_REPORTED), the GPU must stay
usable, and a normal call afterwards must leave the word at zero and match
the oracle.
"""

import ctypes

import pytest
import torch

import oracle
from log_linear_attention_chunkwise_gb300 import binding
from log_linear_attention_chunkwise_gb300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu

LLA_DEVERR_SYNC_TIMEOUT = 2


def _inputs(T=384, H=2):
    cfg = W.small_fwd_config(1, H, T, 128, 128, 64, torch.bfloat16, seed=77)
    x = W.make_fwd_inputs(cfg)
    return x, {n: t.cuda() for n, t in x.items()}


def test_clean_call_leaves_the_word_at_zero():
    x, xd = _inputs()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["lam"], chunk=64, device_error=err)
    assert binding.device_error_check(err) == 0
    assert_parity(out, oracle.naive(x["q"], x["k"], x["v"], x["g"], x["lam"]), torch.bfloat16, "clean")


def test_withheld_product_is_reported_and_the_gpu_recovers():
    x, xd = _inputs()
    lib = binding.load()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.debug_withhold_first_product(True)
    try:
        binding.fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["lam"], chunk=64, device_error=err)
        code = ctypes.c_int32(0)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = lib.lla_device_error_check(ctypes.c_void_p(err.data_ptr()), ctypes.byref(code), stream)
    finally:
        binding.debug_withhold_first_product(False)
    assert rc == 5, binding.STATUS.get(rc, rc)          # LLA_ERR_DEVICE_REPORTED
    assert code.value == LLA_DEVERR_SYNC_TIMEOUT
    # the context is intact: a normal call on the same inputs is correct and clean
    err.zero_()
    out = binding.fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["lam"], chunk=64, device_error=err)
    assert binding.device_error_check(err) == 0
    assert_parity(out, oracle.naive(x["q"], x["k"], x["v"], x["g"], x["lam"]), torch.bfloat16,
                  "after the withheld call")


def test_host_and_noalloc_entry_points_report_too():
    x, xd = _inputs(T=256, H=1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hx = {n: t.pin_memory() for n, t in x.items()}
    binding.debug_withhold_first_product(True)
    try:
        binding.fwd_host(hx["q"], hx["k"], hx["v"], hx["g"], hx["lam"], chunk=64, device_error=err)
        host_code = binding.device_error_check(err)
        err.zero_()
        lib = binding.load()
        out = torch.empty((1, 1, 256, 128), device="cuda")
        p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = lib.lla_fwd_noalloc(p(xd["q"]), p(xd["k"]), p(xd["v"]), p(xd["g"]), p(xd["lam"]), p(out),
                                 1, 1, 256, 128, 128, 64, 1, 0, p(err), stream)
        assert rc == 0
        noalloc_code = binding.device_error_check(err)
    finally:
        binding.debug_withhold_first_product(False)
    assert host_code == LLA_DEVERR_SYNC_TIMEOUT
    assert noalloc_code == LLA_DEVERR_SYNC_TIMEOUT
