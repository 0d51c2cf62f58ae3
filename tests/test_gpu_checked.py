"""The GPU suites once more against the checked build (every global index
and TMA coordinate range-checked in the kernels; a violation raises
DECODE_ATTN_DEV_CHECK and skips the access).  A memory checker cannot run
on these GPUs, so this is how an out-of-range access would show: the suites
assert that no device error bit is set on valid inputs (the two tests that
time a pipeline out on purpose are left out)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_append.py", "tests/test_gpu_multi.py",
          "tests/test_gpu_bf16.py", "tests/test_gpu_cluster.py", "tests/test_gpu_poison.py",
          "tests/test_gpu_invariants.py", "tests/test_gpu_random.py",
          "tests/test_gpu_properties_random.py"]


def test_gpu_suites_pass_on_the_checked_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if os.environ.get("DECODE_ATTN_CHECKED") == "1":
        pytest.skip("already running on the checked build")
    env = dict(os.environ, DECODE_ATTN_CHECKED="1")
    probe = subprocess.run(
        [sys.executable, "-c", "from paged_gqa_decode_06_gb300 import build; build.build(); "
         "import paged_gqa_decode_06_gb300 as p; p.load_library(); print(p.library_path())"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.strip().endswith("libpaged_gqa_decode_checked.so")
    r = subprocess.run([sys.executable, "-m", "pytest", "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider", *SUITES, "-k", "not stall"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)
    assert r.returncode == 0, r.stdout[-4000:]
    assert " passed" in r.stdout
