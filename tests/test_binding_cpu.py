"""The Python binding only marshals device tensors into the C ABI: handed host
tensors, every device entry point refuses them before any library call (no
host fallback computes anything).  Runs without a GPU."""

import os

import pytest
import torch

from log_linear_attention_chunkwise_gb300 import binding


@pytest.fixture(scope="module", autouse=True)
def built_library():
    # some entry points load the library before looking at their arguments
    if not os.path.exists(binding.LIB_PATH):
        from log_linear_attention_chunkwise_gb300 import build
        build.build()

B, H, T, D = 1, 2, 64, 16
L = 1 + (T - 1).bit_length()  # levels of T tokens


def host(*shape, dtype=torch.float32):
    return torch.zeros(shape, dtype=dtype)


CALLS = {
    "fwd": lambda: binding.fwd(host(B, H, T, D), host(B, H, T, D), host(B, H, T, D), host(B, H, T),
                               host(B, H, T, L)),
    "bwd": lambda: binding.bwd(host(B, H, T, D), host(B, H, T, D), host(B, H, T, D), host(B, H, T),
                               host(B, H, T, L), host(B, H, T, D)),
    "gdn_fwd": lambda: binding.gdn_fwd(host(B, H, T, D), host(B, H, T, D), host(B, H, T, D), host(B, H, T),
                                       host(B, H, T), host(B, H, T, L)),
    "gdn_decode_step": lambda: binding.gdn_decode_step(host(B, H, 4, D, D), host(B, H, D), host(B, H, D),
                                                       host(B, H, D), host(B, H), host(B, H), host(B, H, 5),
                                                       host(B, dtype=torch.int64)),
    "decode_step": lambda: binding.decode_step(host(B, H, 4, D, D), host(B, H, 4), host(B, H, D), host(B, H, D),
                                               host(B, H, D), host(B, H), host(B, H, 5),
                                               host(B, dtype=torch.int64)),
    "prefill_state": lambda: binding.prefill_state(host(B, H, T, D), host(B, H, T, D), host(B, H, T), Ls=8),
    "lambda_mlp": lambda: binding.lambda_mlp(host(B, H, T, D), host(D, 2 * L), host(2 * L, L), host(L)),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused(name):
    with pytest.raises(ValueError, match="CUDA tensor"):
        CALLS[name]()
