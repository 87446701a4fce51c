"""Helpers shared by the GPU parity tests (inputs, tolerance checks)."""
import functools

import numpy as np
import pytest

import qsynth

GEMV_TOL_REL = 1e-3      # |y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-6 per element
GEMV_TOL_ABS = 1e-6


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def qlib():
    from block_quantized_weight_qgemv_gb300 import build
    build.build()
    import block_quantized_weight_qgemv_gb300 as q
    q.lib()
    return q


@functools.lru_cache(maxsize=8)
def weights(fmt, nrows, ncols, seed):
    return qsynth.make_weights(fmt, nrows, ncols, seed)


def to_dev(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev(bits, torch):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def assert_within_bound(got, ref, absdot, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = GEMV_TOL_REL * np.asarray(absdot) + GEMV_TOL_ABS
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d elements outside |err| <= 1e-3*sum|w x| + 1e-6; first %s "
                             "got %s ref %s bound %s" % (what, int(bad.sum()), bad.size, idx.tolist(),
                                                         got[bad][:5], ref[bad][:5], bound[bad][:5]))
    return float((err / bound).max()) if err.size else 0.0
