"""The bounds-check build (libqoq_debug.so, loaded when QOQ_DEBUG=1).

In it every GEMM kernel tests each weight-block copy, each split-tile slot
and arrival-counter access and each output element it writes by plain
stores, and the KV4 attention each output and split partial it writes,
against the extent of the buffer; an access outside it is skipped and sets
status bit 8.  This test re-runs, in a child process that loads that
library, the parity suites of all three GEMM paths (every tile size,
schedule, CTA count and split-tile completion route), the KV4 append and
attention suites and the allocation-free entry point.  Each of them compares
with the oracle and, where it reads the status word, requires QOQ_OK, so a
checked access found outside its buffer fails them.  No test plants an
out-of-range access on the GPU.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SELECTION = [
    "tests/test_abi.py::test_loaded_library_matches_request",
    "tests/test_gpu_parity.py",
    "tests/test_gpu_kv4.py",
    "tests/test_zz_no_alloc.py",
]


def test_parity_suites_pass_under_the_bounds_check_build():
    env = dict(os.environ, QOQ_DEBUG="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", *SELECTION],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = r.stdout[-4000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
