"""The debug build: every kernel checks its computed global-memory accesses against the extents of
the tensors it addresses (compiled in with -DGBQ_DEBUG_BOUNDS).  A violation sets GBQ_DEV_BOUNDS in
the device status word and skips the access; nothing traps.  This runs the GPU parity tests (all but
the full-size ones) against libgbq_debug.so in a child process; each of them asserts afterwards that
the device status word is clean, so any out-of-range access fails it."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

SUITE = ["test_gpu_rotate.py", "test_gpu_linear.py", "test_gpu_ffn.py", "test_gpu_backward.py",
         "test_gpu_bf16_path.py", "test_gpu_descriptors.py", "test_gpu_graphs.py", "test_zz_no_alloc.py"]


def test_gpu_suite_under_bounds_checks():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ffn_rotate_quantize_gb300.build import build_lib
    lib = build_lib(debug=True)
    env = dict(os.environ, GBQ_LIB=lib)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"] + \
          [os.path.join(ROOT, "tests", f) for f in SUITE]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-15:])
    assert r.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail, tail
    print(tail.splitlines()[-1])
