"""The index-checked build of the library (compiled with -DTV_DEBUG:
libtv_debug.so).  Compute-sanitizer is not available on the GPU pool, so this
build stands in for a memory checker: before every global-memory access whose
index a kernel computes, it tests that the index lies in its array, records a
failure (tv_debug_check_failures) and skips the access.

The test builds it, then runs the GPU test files on it in a child process
(TV_LIB_PATH selects the library): every test must pass, and at the end of
that session no index check may have failed (tests/conftest.py).  The
full-size sampled cases are left out for time; every small parity case, the
bad-input cases, the graph replays, the no-allocation entry point and the
bounded-wait expiry cases run."""
import os
import re
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["tests/test_gpu_parity.py", "tests/test_gpu_draft.py", "tests/test_gpu_gdn.py",
         "tests/test_gpu_graph.py", "tests/test_zy_expiry.py", "tests/test_zz_no_alloc.py"]


def test_gpu_suite_on_the_index_checked_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    lib = __graft_entry__._builder().build(debug=True)
    env = dict(os.environ, TV_LIB_PATH=lib, TV_DEBUG_CHECKS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "-k", "not full_size", *FILES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = (r.stdout[-4000:] + "\n" + r.stderr[-2000:])
    assert r.returncode == 0, tail
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 150, tail  # the small cases ran, not a filtered-out session
