"""Child process of test_gpu_gemm_paths.py: prefill parity checks with the
kernel choice forced by QGEMV_GEMM_PATH."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
import qsynth  # noqa: E402
from gpu_util import assert_within_bound, bf16_dev, qlib  # noqa: E402

CASES = [("q4_0", 200, 320, 77), ("q4_1", 129, 256, 130), ("q8_0", 400, 512, 33)]


def main():
    q = qlib()
    oracle.build()
    for fmt, nrows, ncols, m in CASES:
        Wn = qsynth.make_weights(fmt, nrows, ncols, seed=nrows)
        Xn = qsynth.make_X_bf16(m, ncols, seed=m)
        W = torch.from_numpy(Wn).cuda()
        X = bf16_dev(Xn, torch)
        Y = torch.full((m, nrows), float("nan"), device="cuda")
        getattr(q, "qgemm_" + fmt)(W, X, Y, nrows, ncols, m)
        torch.cuda.synchronize()
        q.qgemv_sync_check()
        ref, ab = oracle.gemm(fmt, Wn, Xn, nrows, ncols, m)
        assert_within_bound(Y.cpu().numpy(), ref, ab, "%s %s" % (os.environ.get("QGEMV_GEMM_PATH"), fmt))
    print("ok")


if __name__ == "__main__":
    main()
