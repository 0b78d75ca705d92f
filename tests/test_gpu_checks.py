"""The build with internal bounds checks (libcsa_checks.so, CSA_CHECKS=1).

Every bounds check inside the library must hold on the parity and full-size
workloads: the GPU parity, HCA, sharded-decode and FP4 tests run again in a
child process that loads the checked build, and they require a zero status word (a failed check would set
CSA_DEV_CHECK) besides their usual comparisons with the oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_under_the_checked_build(cuda_device):
    from sparse_compressed_kv_gb300 import build as B
    B.build(checks=True)
    env = dict(os.environ, CSA_CHECKS="1")
    which = subprocess.run([sys.executable, "-c", "from sparse_compressed_kv_gb300 import csa; "
                            "csa.load(); print(csa.LIB_PATH)"], cwd=ROOT, env=env,
                           capture_output=True, text=True, timeout=300)
    assert which.stdout.strip().endswith("libcsa_checks.so"), which.stdout + which.stderr
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join("tests", "test_gpu_parity.py"), os.path.join("tests", "test_gpu_hca.py"),
           os.path.join("tests", "test_gpu_shard.py"), os.path.join("tests", "test_gpu_fp4.py"),
           os.path.join("tests", "test_gpu_full_size.py") + "::test_batch32_decode"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
