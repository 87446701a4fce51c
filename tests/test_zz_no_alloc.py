"""qgemm_q4_0_noalloc: the Q4_0 prefill for callers that cannot let a library
allocate device memory (memory reserved up front, or no tolerance for the
synchronization an allocation can imply).  Its activation copy lives in a
fixed 8 MiB device array of the library instead of a grown workspace.

Called through the C ABI; on two calls in a row (different inputs and shapes,
so the second call reuses the array the first one filled) its output must
match the existing qgemm_q4_0 entry point within the prefill tolerance
(|dY| <= 1e-3 * sum_k |w_k x_k| + 1e-6, the sum taken from the CPU oracle).
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import qsynth
from gpu_util import assert_within_bound, bf16_dev, qlib, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def _call(fn, torch, W, X, Y, nrows, ncols, m):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.c_void_p(W.data_ptr()), ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(Y.data_ptr()),
              nrows, ncols, m, stream)


def _both(q, torch, nrows, ncols, m, seed):
    lib = q.lib()
    Wn = qsynth.make_weights("q4_0", nrows, ncols, seed)
    Xn = qsynth.make_X_bf16(m, ncols, seed + 1)
    W = to_dev(Wn, torch)
    X = bf16_dev(Xn, torch)
    Y_new = torch.full((m, nrows), float("nan"), device="cuda")
    Y_old = torch.full((m, nrows), float("nan"), device="cuda")
    rc = _call(lib.qgemm_q4_0_noalloc, torch, W, X, Y_new, nrows, ncols, m)
    assert rc == 0, lib.qgemv_last_error_string()
    rc = _call(lib.qgemm_q4_0, torch, W, X, Y_old, nrows, ncols, m)
    assert rc == 0, lib.qgemv_last_error_string()
    torch.cuda.synchronize()
    assert lib.qgemv_sync_check() == 0
    return Wn, Xn, Y_new.cpu().numpy(), Y_old.cpu().numpy()


def test_noalloc_matches_existing_entry_small(oracle_mod):
    torch = torch_cuda()
    q = qlib()
    for (nrows, ncols, m, seed) in [(200, 320, 77, 11), (257, 512, 130, 12)]:    # two calls in a row
        Wn, Xn, y_new, y_old = _both(q, torch, nrows, ncols, m, seed)
        ref, ab = oracle_mod.gemm("q4_0", Wn, Xn, nrows, ncols, m)
        assert_within_bound(y_new, ref, ab, "noalloc vs oracle %dx%d m=%d" % (nrows, ncols, m))
        assert_within_bound(y_new, y_old, ab, "noalloc vs qgemm_q4_0 %dx%d m=%d" % (nrows, ncols, m))


def test_noalloc_matches_existing_entry_prefill_size(oracle_mod):
    """The 512-token prefill of a 14336 x 4096 Q4_0 matrix (4 MiB of scratch),
    twice in a row with different activations."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, m = 14336, 4096, 512
    g = qsynth.rng(99)
    cols = np.sort(g.choice(nrows, 256, replace=False))
    mi = np.repeat(np.arange(0, m, 4), cols.size)
    ni = np.tile(cols, m // 4)
    for seed in (21, 22):
        Wn, Xn, y_new, y_old = _both(q, torch, nrows, ncols, m, seed)
        assert np.all(np.isfinite(y_new))
        ref_s, ab_s = oracle_mod.gemm_entries("q4_0", Wn, Xn, nrows, ncols, m, mi, ni)
        assert_within_bound(y_new[mi, ni], ref_s, ab_s, "noalloc vs oracle (sampled)")
        assert_within_bound(y_new[mi, ni], y_old[mi, ni], ab_s, "noalloc vs qgemm_q4_0 (sampled)")
        # the two entry points run the same kernel on the same operands
        assert np.array_equal(y_new.view(np.uint32), y_old.view(np.uint32))


def test_noalloc_rejects_problems_beyond_its_scratch():
    torch = torch_cuda()
    q = qlib()
    lib = q.lib()
    nrows, ncols, m = 64, 4096, 1025           # 1025 * 4096 * 2 bytes > 8 MiB
    W = torch.zeros(nrows * ncols // 32 * 18, dtype=torch.uint8, device="cuda")
    X = torch.zeros(m, ncols, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(m, nrows, device="cuda")
    rc = _call(lib.qgemm_q4_0_noalloc, torch, W, X, Y, nrows, ncols, m)
    assert rc == 2
    assert b"scratch" in lib.qgemv_last_error_string()
