"""The CUDA-core prefill kernel (an independent cross-check of the tensor-core
kernel) is parity-checked too, by forcing it in a child process."""
import os
import subprocess
import sys

import pytest

from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("path", ["simple", "tc"])
def test_forced_gemm_path_matches_oracle(path):
    torch_cuda()
    env = dict(os.environ, QGEMV_GEMM_PATH=path)
    r = subprocess.run([sys.executable, os.path.join(HERE, "gemm_path_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
