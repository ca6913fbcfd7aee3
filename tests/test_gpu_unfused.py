"""The separate-kernel path of ffn_swiglu and moe_ffn (router GEMV, gate/up,
down as three launches), which the library takes when a layer does not fit
the fused kernel.  QMOE_FUSED=0 forces it; the switch is read once per
process, so the parity tests run again in a child process with it set."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_separate_kernel_path_parity():
    env = dict(os.environ, QMOE_FUSED="0")
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"),
           os.path.join(ROOT, "tests", "test_gpu_rmsnorm.py"),
           "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
           "-k", "ffn_small or ffn_dense or moe_small or moe_decode or rmsnorm"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
