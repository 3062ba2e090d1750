"""The parity suites again, on the bounds-check build of the library (the
same sources compiled with LLAMA_BOUNDS_CHECK: every kernel checks its
shared-memory layout against the launch's dynamic shared memory and its index
invariants, and a failure sets LLAMA_FLAG_INDEX, which the suites' status
checks turn into a failure). This stands in for a memory checker: the runs
must pass unchanged, with no index flag."""
import os
import subprocess
import sys

import pytest

from _common import need_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_ops.py", "tests/test_gpu_model.py", "tests/test_gpu_extend.py",
          "tests/test_gpu_sample.py", "tests/test_gpu_fp8.py", "tests/test_gpu_w8.py"]


def _env():
    env = dict(os.environ)
    env["LLAMA_GB300_BOUNDS_CHECK"] = "1"
    return env


def test_parity_suites_pass_on_the_bounds_check_build():
    need_gpu()
    from llama2_decoder_forward_gb300 import build as b
    b.build_library(checked=True)
    probe = subprocess.run(
        [sys.executable, "-c", "from llama2_decoder_forward_gb300 import binding; "
         "print(binding.lib().llama_bounds_checked())"],
        cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip() == "1", probe.stdout + probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", *SUITES],
                       cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
