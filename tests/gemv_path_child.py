"""Child process of test_gpu_gemv_paths.py: runs GEMV parity checks with the
kernel choice forced by QGEMV_GEMV_PATH (read once per process)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
import qsynth  # noqa: E402
from gpu_util import assert_within_bound, qlib  # noqa: E402

CASES = [("q4_0", 4096, 14336, 1), ("q4_0", 14336, 4096, 2), ("q4_1", 300, 4096, 1), ("q4_0", 77, 2048, 8),
         ("q4_1", 4096, 4096, 5), ("q8_0", 1000, 2048, 1), ("q4_0", 16, 256, 3), ("q4_0", 153, 512, 1)]


def main():
    q = qlib()
    oracle.build()
    for fmt, nrows, ncols, batch in CASES:
        Wn = qsynth.make_weights(fmt, nrows, ncols, seed=nrows + ncols)
        xn = qsynth.make_x(batch, ncols, seed=batch)
        W = torch.from_numpy(Wn).cuda()
        x = torch.from_numpy(xn).cuda()
        y = torch.full((batch, nrows), float("nan"), device="cuda")
        getattr(q, "qgemv_" + fmt)(W, x, y, nrows, ncols, batch)
        torch.cuda.synchronize()
        q.qgemv_sync_check()
        ref, ab = oracle.gemv(fmt, Wn, xn, nrows, ncols, batch)
        assert_within_bound(y.cpu().numpy(), ref, ab, "%s %s %dx%d b%d" % (
            os.environ.get("QGEMV_GEMV_PATH"), fmt, nrows, ncols, batch))
    print("ok")


if __name__ == "__main__":
    main()
