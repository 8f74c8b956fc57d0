import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def mr():
    """The CUDA library's Python binding; only usable where a GPU is present."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_gating_expert_row_gb300 as m

    return m


def pytest_terminal_summary(terminalreporter):
    parity = sys.modules.get("parity")
    rows = getattr(parity, "NEAR_TIES", None)
    if not rows:
        return
    terminalreporter.section("near ties at the selection boundary (< 4 fp32 ulp; informational)")
    for what, n, total in rows:
        terminalreporter.write_line(f"{what}: {n} of {total} token rows")
