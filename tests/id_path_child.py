"""Child process of test_gpu_id.py: expert-selected GEMV parity with the
kernel forced by QGEMV_ID_PATH (read once per process).  Shapes the forced
kernel cannot take report QGEMV_ERR_UNIMPLEMENTED (tensor cores: ncols not a
multiple of 1024) and are skipped; the general kernel takes every shape."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
import qsynth  # noqa: E402
from gpu_util import assert_within_bound, qlib  # noqa: E402

# (fmt, nrows, ncols, n_expert, ids, x_group)
CASES = [("q4_0", 4096, 14336, 8, [6, 1], 1), ("q4_1", 300, 4096, 8, [3, 5, 3, 0], 2),
         ("q8_0", 77, 2048, 4, [1, 1, 1, 1, 1, 2], 3), ("q4_0", 64, 256, 2, [1], 1),
         ("q4_0", 1000, 4096, 8, [0, 1, 0, 1, 2, 1, 3, 0, 4, 0, 5, 0, 6, 7, 0, 0], 2),
         ("q8_0", 4096, 14336, 8, [3, 3, 3, 3, 3, 3, 3, 3, 3, 1], 1)]


def main():
    q = qlib()
    oracle.build()
    path = os.environ.get("QGEMV_ID_PATH")
    ran = 0
    for fmt, nrows, ncols, n_expert, ids, xg in CASES:
        batch = len(ids)
        Wn = qsynth.make_weights(fmt, n_expert * nrows, ncols, seed=nrows + ncols)
        xn = qsynth.make_x(batch // xg, ncols, seed=batch)
        idsn = np.asarray(ids, np.int32)
        W = torch.from_numpy(Wn).cuda()
        x = torch.from_numpy(xn).cuda()
        idd = torch.from_numpy(idsn).cuda()
        y = torch.full((batch, nrows), float("nan"), device="cuda")
        try:
            getattr(q, "qgemv_id_" + fmt)(W, n_expert, idd, x, y, nrows, ncols, batch, x_group=xg)
        except q.QgemvError as e:
            if path == "tc" and e.status == 9:
                continue
            raise
        torch.cuda.synchronize()
        q.qgemv_sync_check()
        ref, ab = oracle.gemv_id(fmt, Wn, n_expert, idsn, xn, nrows, ncols, batch, xg)
        assert_within_bound(y.cpu().numpy(), ref, ab, "%s %s %dx%d" % (path, fmt, nrows, ncols))
        ran += 1
    assert ran >= 5, ran
    print("ok")


if __name__ == "__main__":
    main()
