"""Child process of test_gpu_mmvq.py: quantized-activation GEMV parity with the
kernel forced by QGEMV_MMVQ_PATH (read once per process).  Shapes the forced
kernel cannot take are skipped for the streaming kernel (the call reports
QGEMV_ERR_UNIMPLEMENTED) and run everywhere for the general one."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
import qsynth  # noqa: E402
from gpu_util import qlib  # noqa: E402
from test_gpu_mmvq import assert_mmvq_close  # noqa: E402

CASES = [("q4_0", 4096, 14336, 1), ("q4_0", 14336, 4096, 2), ("q4_1", 300, 4096, 8), ("q8_0", 77, 2048, 3),
         ("q8_0", 1000, 14336, 5), ("q4_1", 33, 128, 1), ("q4_0", 16, 256, 6), ("q4_0", 5, 96, 2)]


def main():
    q = qlib()
    oracle.build()
    path = os.environ.get("QGEMV_MMVQ_PATH")
    ran = 0
    for fmt, nrows, ncols, batch in CASES:
        Wn = qsynth.make_weights(fmt, nrows, ncols, seed=nrows + ncols)
        xn = qsynth.make_x(batch, ncols, seed=batch)
        W = torch.from_numpy(Wn).cuda()
        x = torch.from_numpy(xn).cuda()
        y = torch.full((batch, nrows), float("nan"), device="cuda")
        try:
            getattr(q, "qgemv_mmvq_" + fmt)(W, x, y, nrows, ncols, batch)
        except q.QgemvError as e:
            if path == "stream" and e.status == 9:
                continue
            raise
        torch.cuda.synchronize()
        q.qgemv_sync_check()
        rq, rd, _ = oracle.quantize_q8_1(xn, ncols, batch)
        ref, ab = oracle.gemv_q8_1(fmt, Wn, rq, rd, nrows, ncols, batch)
        assert_mmvq_close(y.cpu().numpy(), ref, ab, "%s %s %dx%d b%d" % (path, fmt, nrows, ncols, batch))
        ran += 1
    assert ran >= 6, ran
    print("ok")


if __name__ == "__main__":
    main()
