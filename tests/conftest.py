"""Test configuration: the `gpu` marker and shared fixtures.

`-m "not gpu"` runs the oracle pins, the host-side logic and the C-ABI
load/export checks on CPU.  `-m gpu` runs the parity tests, which call the
CUDA library through the C ABI and compare with the CPU oracle.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def qm():
    """The CUDA library, built in-tree and loaded (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_ffn_gb300 as qm
    qm.build()
    qm.lib()
    # child test processes of test_gpu_unfused.py run the suite in one of the
    # library's other kernel forms
    mode = os.environ.get("QMOE_TEST_EXEC_MODE")
    if mode:
        qm.set_exec_mode(int(mode))
    return qm
