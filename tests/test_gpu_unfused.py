"""Paths the library takes only when the default one does not apply, run in
child processes whose qm fixture selects them with qmoe_set_exec_mode (the
test harness passes the mode in QMOE_TEST_EXEC_MODE; the library reads no
environment):
  - QMOE_EXEC_SEPARATE: the separate-kernel form of ffn_swiglu and moe_ffn
    (router GEMV, gate/up, down as three launches), taken when a layer does
    not fit the fused kernel;
  - QMOE_EXEC_UNBATCHED: 2..31 tokens as one fused launch per token, taken
    when the batched kernel's tiles do not fit shared memory."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_separate_kernel_path_parity():
    env = dict(os.environ, QMOE_TEST_EXEC_MODE="1")
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"),
           os.path.join(ROOT, "tests", "test_gpu_rmsnorm.py"),
           "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
           "-k", "ffn_small or ffn_dense or moe_small or moe_decode or rmsnorm or no_renorm "
           "or non_finite"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


@pytest.mark.gpu
def test_token_by_token_path_parity():
    env = dict(os.environ, QMOE_TEST_EXEC_MODE="2")
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_batch.py"),
           os.path.join(ROOT, "tests", "test_gpu_rmsnorm.py"),
           os.path.join(ROOT, "tests", "test_gpu_parity.py"),
           "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
           "-k", "all_tokens or moe_ffn_rmsnorm or non_finite"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
