"""Tolerances of the GPU-vs-oracle parity tests.

bf16 inputs with fp32 accumulation: max |gpu - oracle| <= 2e-2 and
||gpu - oracle||_F / ||oracle||_F <= 5e-3 over the compared elements.
fp32 inputs: ||gpu - oracle||_F / ||oracle||_F <= 1e-4 and
max |gpu - oracle| <= 1e-4 * max |oracle|.
The oracle reads the same rounded inputs the GPU reads, promoted exactly to
fp64, so the comparison measures the kernels' arithmetic only.

Stress variants (gates forced to 0 on some heads, so nothing decays and the
outputs grow with the sequence length) keep the relative Frobenius bound and
take the max-abs bound relative to the output's magnitude:
max |gpu - oracle| <= max(2e-2, 5e-3 * max |oracle|).  The bf16 operands of
the tensor-core products carry a relative rounding of 2^-9, so an absolute
bound cannot hold for outputs of arbitrary magnitude.
"""

import numpy as np
import torch

# (what, max_abs, rel_fro, max |oracle|, stress) of every comparison made in
# this process; conftest prints them at the end of the run
RECORDS = []

BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 5e-3
F32_REL_FRO = 1e-4
F32_REL_MAX = 1e-4


def errors(gpu, ref):
    g = gpu.detach().to("cpu").double().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    d = g - r
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    ref_fro = float(np.linalg.norm(r))
    rel_fro = float(np.linalg.norm(d)) / ref_fro if ref_fro > 0 else float(np.linalg.norm(d))
    ref_max = float(np.max(np.abs(r))) if r.size else 0.0
    return max_abs, rel_fro, ref_max


def assert_parity(gpu, ref, in_dtype, what="", stress=False):
    max_abs, rel_fro, ref_max = errors(gpu, ref)
    RECORDS.append((what, max_abs, rel_fro, ref_max, stress, in_dtype == torch.bfloat16))
    if in_dtype == torch.bfloat16:
        amax = max(BF16_MAX_ABS, BF16_REL_FRO * ref_max) if stress else BF16_MAX_ABS
        ok = max_abs <= amax and rel_fro <= BF16_REL_FRO
        bound = f"max_abs<={amax:.3g}, rel_fro<={BF16_REL_FRO}"
    else:
        ok = rel_fro <= F32_REL_FRO and max_abs <= F32_REL_MAX * max(ref_max, 1e-30)
        bound = f"rel_fro<={F32_REL_FRO}, max_abs<={F32_REL_MAX}*{ref_max:.3g}"
    assert ok, f"{what}: max_abs={max_abs:.3e} rel_fro={rel_fro:.3e} ({bound})"
    return max_abs, rel_fro
