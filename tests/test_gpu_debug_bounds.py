"""The bounds-checked build of the library (-DMOE_DEBUG_BOUNDS: every slot,
key, pair position, h row and output row the kernels derive is checked
before use, violations counted and skipped) runs the decode, prefill, W4A4,
graph and failure-path GPU tests without a single violation.  This is the
stand-in for a device memory checker; the tests also check their results, so
a skipped access would show up as a parity failure too."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_build_runs_the_gpu_tests_without_violations():
    from expert_cache_serving_gb300 import build as b

    lib = b.build_cuda(debug=True)
    env = dict(os.environ, MOECACHE_LIB=lib, MOE_EXPECT_DEBUG="1")
    tests = ["tests/test_gpu_decode.py", "tests/test_gpu_prefill.py", "tests/test_gpu_w4a4.py",
             "tests/test_gpu_graph.py", "tests/test_gpu_failure_paths.py", "tests/test_gpu_qstar.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider"] + tests,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=2400)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
