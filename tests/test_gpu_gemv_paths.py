"""Every GEMV kernel is parity-checked, whichever one the dispatch would pick:
each case runs in a child process with QGEMV_GEMV_PATH forcing the fixed-point
dp4a kernel, the stream-K tensor-core kernel, the streamed CUDA-core kernel or
the warp-per-row kernel (a kernel that cannot take a shape falls back to the
next, so all shapes still run)."""
import os
import subprocess
import sys

import pytest

from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("path", ["fx", "sk", "stream", "rowwarp"])
def test_forced_gemv_path_matches_oracle(path):
    torch_cuda()
    env = dict(os.environ, QGEMV_GEMV_PATH=path)
    r = subprocess.run([sys.executable, os.path.join(HERE, "gemv_path_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
