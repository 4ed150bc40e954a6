"""The map, shape, fit and attention parity tests on the checked build.

libkvb_checked.so is the library compiled with KVB_CHECK_BOUNDS=1: every
CUDA-core global access of the hot kernels (the map epilogue's bias reads and
stores, the fused and standalone key strips, the four-matrix calibration
gather's stores, the statistics merge's read-modify-writes, the attention
cosines) first checks its index range against its buffer; a failed check
records an error code instead of touching memory, and the next call on the
context (or kvb_ctx_check) returns KVB_ERR_CUDA.  The same parity tests that
run on the normal library then pass only if no such access strayed.  It stands
in for a memory checker, which is not available on these GPUs.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_map.py", "tests/test_gpu_shapes.py", "tests/test_gpu_fit.py",
          "tests/test_gpu_attention.py"]


def test_parity_suites_pass_on_the_checked_build():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cross_model_kv_gb300 import build
    build.build(checked=True)
    env = dict(os.environ, KVB_LIBRARY="checked")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-2000:])
    assert " passed" in r.stdout
