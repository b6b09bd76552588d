import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built liblla.so")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("test marked gpu but no CUDA device is visible")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Measured parity errors: the largest max-abs of the bf16 comparisons,
    and every stress comparison beside the absolute 2e-2 bound of the
    workloads (stress cases are judged on max(2e-2, 5e-3 max|oracle|))."""
    try:
        from parity import RECORDS
    except ImportError:
        return
    bf16 = [r for r in RECORDS if r[5]]
    if not bf16:
        return
    tr = terminalreporter
    tr.section("parity errors (bf16 inputs)")
    worst = max((r for r in bf16 if not r[4]), key=lambda r: r[1], default=None)
    if worst:
        tr.write_line(f"largest max_abs outside stress cases: {worst[1]:.3e} ({worst[0]}), "
                      f"rel_fro {worst[2]:.2e}")
    for what, max_abs, rel_fro, ref_max, stress, _ in bf16:
        if stress:
            tr.write_line(f"stress {what}: max_abs {max_abs:.3e} ({max_abs / 2e-2:.2f} x 2e-2), "
                          f"rel_fro {rel_fro:.2e}, max|oracle| {ref_max:.3g}")
