"""GPU parity of the prefill matmul against the CPU oracle, through the C ABI.

Bar: |Y_gpu - Y_ref| <= 1e-3 * sum_k |w_k X_k| + 1e-6 for every compared
element.  Small and ragged shapes are compared in full; the 512 x 4096 by
14336 x 4096 Q4_0 prefill (the benchmark's launch configuration) is compared
on all 512 token rows for a seeded sample of 1024 output columns."""
import numpy as np
import pytest

import qsynth
from gpu_util import assert_within_bound, bf16_dev, qlib, to_dev, torch_cuda, weights

pytestmark = pytest.mark.gpu

FMTS = ["q4_0", "q4_1", "q8_0"]


def run_gemm(q, torch, fmt, Wn, Xn, nrows, ncols, m):
    W = to_dev(Wn, torch)
    X = bf16_dev(Xn, torch)
    Y = torch.full((m, nrows), float("nan"), dtype=torch.float32, device="cuda")
    getattr(q, "qgemm_" + fmt)(W, X, Y, nrows, ncols, m)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    return Y.cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(64, 256, 8), (128, 128, 128), (200, 320, 77), (1, 64, 1),
                                   (257, 512, 130), (96, 1024, 300)])
def test_gemm_small(oracle_mod, fmt, shape):
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, m = shape
    Wn = weights(fmt, nrows, ncols, 50 + nrows)
    Xn = qsynth.make_X_bf16(m, ncols, 51 + m)
    got = run_gemm(q, torch, fmt, Wn, Xn, nrows, ncols, m)
    ref, ab = oracle_mod.gemm(fmt, Wn, Xn, nrows, ncols, m)
    assert_within_bound(got, ref, ab, "%s %s" % (fmt, shape))


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_prefill_full_size_sampled(oracle_mod, fmt):
    """The benchmark's shape in every format: each format's raw-weight ring
    (Q4_0 4-chunk, Q4_1 3-stage, Q8_0 shifted boxes) wraps many times."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, m = 14336, 4096, 512
    Wn = weights(fmt, nrows, ncols, 4000)
    Xn = qsynth.make_X_bf16(m, ncols, 4001)
    got = run_gemm(q, torch, fmt, Wn, Xn, nrows, ncols, m)
    cols = np.sort(qsynth.rng(4002).choice(nrows, 1024, replace=False))
    mi = np.repeat(np.arange(m), cols.size)
    ni = np.tile(cols, m)
    ref, ab = oracle_mod.gemm_entries(fmt, Wn, Xn, nrows, ncols, m, mi, ni)
    assert_within_bound(got[mi, ni], ref, ab, "prefill sampled " + fmt)
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(193, 768, 40), (385, 2304, 257)])
def test_gemm_superchunk_tails(oracle_mod, fmt, shape):
    """Raw-weight rings whose superchunk count is odd or not a power of two
    (Q4_0: 3 and 9 superchunks over 2 stages; Q4_1: 6 and 18 over 3; Q8_0: 6
    and 18 shifted boxes over 2), with ragged row tiles and token groups.
    Column counts off the TMA path (ncols % 256 != 0 for Q4_0 / Q8_0, % 128
    for Q4_1) are in test_gemm_small."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, m = shape
    Wn = weights(fmt, nrows, ncols, 60 + nrows)
    Xn = qsynth.make_X_bf16(m, ncols, 61 + m)
    got = run_gemm(q, torch, fmt, Wn, Xn, nrows, ncols, m)
    ref, ab = oracle_mod.gemm(fmt, Wn, Xn, nrows, ncols, m)
    assert_within_bound(got, ref, ab, "%s %s" % (fmt, shape))


def test_gemm_empty_and_errors():
    torch = torch_cuda()
    q = qlib()
    W = to_dev(weights("q4_0", 4, 128, 1), torch)
    X = torch.zeros(2, 128, dtype=torch.bfloat16, device="cuda")
    Y = torch.full((2, 4), 5.0, device="cuda")
    q.qgemm_q4_0(W, X, Y, 4, 128, 0)
    torch.cuda.synchronize()
    assert torch.all(Y == 5.0)
    with pytest.raises(q.QgemvError) as e:
        q.qgemm_q4_0(W, X, Y, 4, 96, 2)
    assert e.value.status == 2
