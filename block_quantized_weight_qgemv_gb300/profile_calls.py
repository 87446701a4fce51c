"""Runs a few calls of one library entry point on seeded synthetic inputs, for
profiler captures (ncu) of a single kernel:

    python -m block_quantized_weight_qgemv_gb300.profile_calls gemv q4_0 4096 14336 1
    python -m block_quantized_weight_qgemv_gb300.profile_calls dequant q4_0 2048 32768
    python -m block_quantized_weight_qgemv_gb300.profile_calls gemm q4_0 14336 4096 512
    python -m block_quantized_weight_qgemv_gb300.profile_calls packed q4_0 4096 14336 1

gemv: FMT NROWS NCOLS BATCH -- six qgemv calls over four copies of W (so the
captured launch does not find W in L2); dequant: FMT NROWS NCOLS -- four
to-fp16 calls; gemm: FMT NROWS NCOLS M -- four prefill calls; packed: q4_0
NROWS NCOLS BATCH -- four copies of W packed once, then six GEMV calls on them.  Exits 0 after a
synchronize and a qgemv_sync_check.
"""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import qsynth  # noqa: E402

import block_quantized_weight_qgemv_gb300 as q  # noqa: E402


def main(argv):
    what, fmt = argv[0], argv[1]
    dims = [int(v) for v in argv[2:]]
    if what == "gemv":
        nrows, ncols, batch = dims
        Wn = qsynth.make_weights(fmt, nrows, ncols, 1)
        copies = [torch.from_numpy(Wn).cuda() for _ in range(4)]
        x = torch.from_numpy(qsynth.make_x(batch, ncols, 2)).cuda()
        y = torch.empty(batch, nrows, device="cuda")
        for i in range(6):
            getattr(q, "qgemv_" + fmt)(copies[i % 4], x, y, nrows, ncols, batch)
    elif what == "packed":
        nrows, ncols, batch = dims
        W = torch.from_numpy(qsynth.make_weights(fmt, nrows, ncols, 1)).cuda()
        nbytes = q.qgemv_packed_bytes(nrows, ncols)
        copies = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(4)]
        for Wp in copies:
            q.qgemv_pack_q4_0(W, Wp, nrows, ncols)
        del W
        x = torch.from_numpy(qsynth.make_x(batch, ncols, 2)).cuda()
        y = torch.empty(batch, nrows, device="cuda")
        for i in range(6):
            q.qgemv_packed_q4_0(copies[i % 4], x, y, nrows, ncols, batch)
    elif what == "dequant":
        nrows, ncols = dims
        W = torch.from_numpy(qsynth.make_weights(fmt, nrows, ncols, 1)).cuda()
        out = torch.empty(nrows, ncols, dtype=torch.float16, device="cuda")
        for _ in range(4):
            getattr(q, "qdequant_" + fmt)(W, out, nrows, ncols)
    elif what == "gemm":
        nrows, ncols, m = dims
        W = torch.from_numpy(qsynth.make_weights(fmt, nrows, ncols, 1)).cuda()
        X = torch.from_numpy(qsynth.make_X_bf16(m, ncols, 2)).cuda()
        Y = torch.empty(m, nrows, device="cuda")
        for _ in range(4):
            getattr(q, "qgemm_" + fmt)(W, X.view(torch.bfloat16), Y, nrows, ncols, m)
    else:
        raise SystemExit("unknown operation %r" % what)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    print("ok")


if __name__ == "__main__":
    main(sys.argv[1:])
