"""The checking build of the library (libgqa_debug.so: the same kernels with
device bounds checks that set GQA_DEVERR_BOUNDS and skip the access instead
of trapping) on small cases of every kernel family, in a child process so
that it loads that build alone.  It stands in for a memory checker: no index
computed by the kernels may leave its buffer, and the results stay exact to
the oracle's tolerance."""
import os
import subprocess
import sys

import pytest

import grouped_query_decode_kv_b300 as gqa

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_checking_build_small_cases():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    lib = os.path.join(os.path.dirname(gqa.__file__), "libgqa_debug.so")
    if not os.path.exists(lib):
        from grouped_query_decode_kv_b300 import build
        build.build()
    env = dict(os.environ, GQA_LIBRARY=lib, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_cases.py")], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ALL OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
