"""The bounds-checking build: libvsf_bounds.so is libvsf compiled with
-DVSF_DEBUG_BOUNDS, whose kernels check every range they index (tensor
segments, ring chunks, quantisation blocks, 8-element groups, matrices)
against the packed buffers' extent and set bit 4 of the device error word
instead of accessing out of range. It stands in for a memory checker: the
parity, rank-window, group-op, Muon and resume suites run against it in a
child process, and every step (or every ShardStep at close) must leave the
error word clear. The tests marked slow (the largest full-size cases, which
the normal build runs) are left out of the child's run to bound its time;
the Llama layer's and DSv3 block's full-size windows stay in.
"""
import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_rank_window.py",
          "tests/test_gpu_group_ops.py", "tests/test_gpu_muon.py", "tests/test_gpu_resume.py"]


def test_suites_pass_under_the_bounds_checking_build():
    from fsdp_buffer_layout_gb300 import _build
    lib = _build.build(variant="bounds")
    env = dict(os.environ, VSF_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-m", "gpu and not slow", "-x",
                        "-p", "no:cacheprovider"] + SUITES,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    passed = re.search(r"(\d+) passed", r.stdout)
    assert passed and int(passed.group(1)) >= 40, r.stdout[-2000:]  # the suites really ran
