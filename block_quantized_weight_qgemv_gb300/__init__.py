"""Python binding of libqgemv.so: block-quantized (ggml Q4_0 / Q4_1 / Q8_0)
weight dequantization, GEMV and prefill GEMM on one GB300 GPU.

This module only marshals arguments: every step of the computation runs in the
CUDA kernels of ``libqgemv.so`` (built in-tree by ``build.py``).  There is no
CPU or PyTorch fallback; if the library is missing or cannot be loaded,
importing the functions raises.

Function names follow the C ABI (``include/qgemv.h``).  Tensors are torch CUDA
tensors owned by the caller:

* ``W``: uint8, the packed blocks (``nrows * ncols/32 * block_bytes`` bytes);
* ``x``: float32 ``[batch][ncols]``;  ``y``: float32 ``[batch][nrows]``;
* ``X``: bfloat16 ``[m][ncols]``;  ``Y``: float32 ``[m][nrows]``;
* ``out``: float32 or float16 ``[nrows][ncols]``;
* ``xq``: uint8, quantized activations (``q8_1_size(ncols, batch)`` bytes:
  int8 codes ``[batch][ncols]``, then fp32 scales and int32 code sums
  ``[batch][ncols/32]`` each);
* ``ids``: int32 ``[batch]``, the expert of each output column of an
  expert-selected GEMV (``W`` then holds ``n_expert`` matrices).

``stream`` defaults to torch's current stream on the tensors' device.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "QgemvError", "lib", "BLOCK_BYTES", "QK", "MAX_BATCH", "F32", "F16",
    "qdequant_q4_0", "qdequant_q4_1", "qdequant_q8_0",
    "qgemv_q4_0", "qgemv_q4_1", "qgemv_q8_0",
    "qgemm_q4_0", "qgemm_q4_1", "qgemm_q8_0", "qgemm_q4_0_noalloc",
    "q8_1_size", "q8_1_views", "qquantize_q8_1",
    "qgemv_mmvq_q4_0", "qgemv_mmvq_q4_1", "qgemv_mmvq_q8_0",
    "qgemv_mmvq_xq_q4_0", "qgemv_mmvq_xq_q4_1", "qgemv_mmvq_xq_q8_0",
    "qgemv_id_q4_0", "qgemv_id_q4_1", "qgemv_id_q8_0", "MAX_ID_BATCH",
    "qgemv_sync_check", "qgemv_version", "qgemv_shutdown", "qgemv_set_option",
    "OPT_WEIGHTS_STATIC", "OPT_WAIT_PROBES", "OPT_TEST_WITHHOLD_COPY", "STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemv.so")

QK = 32
MAX_BATCH = 8
MAX_ID_BATCH = 64
F32, F16 = 0, 1
OPT_WEIGHTS_STATIC = 1
OPT_WAIT_PROBES = 2
OPT_TEST_WITHHOLD_COPY = 3
BLOCK_BYTES = {"q4_0": 18, "q4_1": 20, "q8_0": 34, "q4_0_noalloc": 18}
STATUS = {
    0: "QGEMV_OK", 1: "QGEMV_ERR_NULL", 2: "QGEMV_ERR_SHAPE", 3: "QGEMV_ERR_BATCH",
    4: "QGEMV_ERR_ALIGN", 5: "QGEMV_ERR_DTYPE", 6: "QGEMV_ERR_ARCH", 7: "QGEMV_ERR_LAUNCH",
    8: "QGEMV_ERR_TIMEOUT", 9: "QGEMV_ERR_UNIMPLEMENTED", 10: "QGEMV_ERR_CUDA",
    11: "QGEMV_ERR_INDEX",
}

# Every symbol the header declares, with its ctypes signature.
_I64, _INT, _P = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
SIGNATURES = {
    "qdequant_q4_0": ([_P, _P, _I64, _I64, _INT, _P], _INT),
    "qdequant_q4_1": ([_P, _P, _I64, _I64, _INT, _P], _INT),
    "qdequant_q8_0": ([_P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_q4_0": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_q4_1": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_q8_0": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemm_q4_0": ([_P, _P, _P, _I64, _I64, _I64, _P], _INT),
    "qgemm_q4_1": ([_P, _P, _P, _I64, _I64, _I64, _P], _INT),
    "qgemm_q8_0": ([_P, _P, _P, _I64, _I64, _I64, _P], _INT),
    "qgemm_q4_0_noalloc": ([_P, _P, _P, _I64, _I64, _I64, _P], _INT),
    "qgemv_q8_1_size": ([_I64, _INT], _I64),
    "qquantize_q8_1": ([_P, _P, _I64, _INT, _P], _INT),
    "qgemv_mmvq_q4_0": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_mmvq_q4_1": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_mmvq_q8_0": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_mmvq_xq_q4_0": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_mmvq_xq_q4_1": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_mmvq_xq_q8_0": ([_P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_id_q4_0": ([_P, _I64, _P, _P, _INT, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_id_q4_1": ([_P, _I64, _P, _P, _INT, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_id_q8_0": ([_P, _I64, _P, _P, _INT, _P, _I64, _I64, _INT, _P], _INT),
    "qgemv_status_string": ([_INT], ctypes.c_char_p),
    "qgemv_last_error_string": ([], ctypes.c_char_p),
    "qgemv_sync_check": ([], _INT),
    "qgemv_version": ([], _INT),
    "qgemv_shutdown": ([], None),
    "qgemv_set_option": ([_INT, _INT], _INT),
}


class QgemvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__("%s: %s%s" % (where, STATUS.get(status, "QGEMV_ERR_UNKNOWN"),
                                       (" (" + detail + ")") if detail else ""))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libqgemv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libqgemv.so is not built (run "
                              "`python -m block_quantized_weight_qgemv_gb300.build`)")
        l = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.argtypes = args
            fn.restype = res
        _lib = l
    return _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise QgemvError(status, where, lib().qgemv_last_error_string().decode(errors="replace"))


_raw_stream_fn = None


def _stream(t, stream):
    """The cudaStream_t to launch on: `stream` (a handle or a torch stream),
    else torch's current stream on t's device.  The raw current-stream getter
    torch keeps for its own launch paths is used when present (a call costs a
    fraction of building a torch.cuda.Stream object); otherwise the public
    torch.cuda.current_stream."""
    global _raw_stream_fn
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    if _raw_stream_fn is None:
        import torch
        fn = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _raw_stream_fn = (lambda dev: fn(dev)) if fn is not None else \
            (lambda dev: torch.cuda.current_stream(dev).cuda_stream)
    return _raw_stream_fn(t.get_device())


def _need(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _dequant(fmt, W, out, nrows, ncols, stream):
    import torch
    _need(W, torch.uint8, "W")
    if out.dtype == torch.float32:
        dt = F32
    elif out.dtype == torch.float16:
        dt = F16
    else:
        raise TypeError("out must be float32 or float16")
    _need(out, out.dtype, "out")
    if W.numel() < nrows * (ncols // QK) * BLOCK_BYTES[fmt] or out.numel() < nrows * ncols:
        raise ValueError("W or out is smaller than nrows x ncols requires")
    fn = getattr(lib(), "qdequant_" + fmt)
    _check(fn(W.data_ptr(), out.data_ptr(), nrows, ncols, dt, _stream(W, stream)), "qdequant_" + fmt)
    return out


def _gemv(fmt, W, x, y, nrows, ncols, batch, stream):
    import torch
    _need(W, torch.uint8, "W")
    _need(x, torch.float32, "x")
    _need(y, torch.float32, "y")
    if (W.numel() < nrows * (ncols // QK) * BLOCK_BYTES[fmt] or x.numel() < batch * ncols
            or y.numel() < batch * nrows):
        raise ValueError("W, x or y is smaller than the problem requires")
    fn = getattr(lib(), "qgemv_" + fmt)
    _check(fn(W.data_ptr(), x.data_ptr(), y.data_ptr(), nrows, ncols, batch, _stream(W, stream)),
           "qgemv_" + fmt)
    return y


def _gemm(fmt, W, X, Y, nrows, ncols, m, stream):
    import torch
    _need(W, torch.uint8, "W")
    _need(X, torch.bfloat16, "X")
    _need(Y, torch.float32, "Y")
    if (W.numel() < nrows * (ncols // QK) * BLOCK_BYTES[fmt] or X.numel() < m * ncols
            or Y.numel() < m * nrows):
        raise ValueError("W, X or Y is smaller than the problem requires")
    fn = getattr(lib(), "qgemm_" + fmt)
    _check(fn(W.data_ptr(), X.data_ptr(), Y.data_ptr(), nrows, ncols, m, _stream(W, stream)),
           "qgemm_" + fmt)
    return Y


def qdequant_q4_0(W, out, nrows, ncols, stream=None):
    return _dequant("q4_0", W, out, nrows, ncols, stream)


def qdequant_q4_1(W, out, nrows, ncols, stream=None):
    return _dequant("q4_1", W, out, nrows, ncols, stream)


def qdequant_q8_0(W, out, nrows, ncols, stream=None):
    return _dequant("q8_0", W, out, nrows, ncols, stream)


def qgemv_q4_0(W, x, y, nrows, ncols, batch, stream=None):
    return _gemv("q4_0", W, x, y, nrows, ncols, batch, stream)


def qgemv_q4_1(W, x, y, nrows, ncols, batch, stream=None):
    return _gemv("q4_1", W, x, y, nrows, ncols, batch, stream)


def qgemv_q8_0(W, x, y, nrows, ncols, batch, stream=None):
    return _gemv("q8_0", W, x, y, nrows, ncols, batch, stream)


def qgemm_q4_0(W, X, Y, nrows, ncols, m, stream=None):
    return _gemm("q4_0", W, X, Y, nrows, ncols, m, stream)


def qgemm_q4_1(W, X, Y, nrows, ncols, m, stream=None):
    return _gemm("q4_1", W, X, Y, nrows, ncols, m, stream)


def qgemm_q8_0(W, X, Y, nrows, ncols, m, stream=None):
    return _gemm("q8_0", W, X, Y, nrows, ncols, m, stream)


def qgemm_q4_0_noalloc(W, X, Y, nrows, ncols, m, stream=None):
    """Q4_0 prefill that allocates nothing: its activation copy uses a fixed
    8 MiB device array of the library (m * ncols * 2 bytes at most).  For
    callers that cannot let a library allocate device memory."""
    return _gemm("q4_0_noalloc", W, X, Y, nrows, ncols, m, stream)


def q8_1_size(ncols: int, batch: int) -> int:
    """Bytes of the quantized activations of `batch` columns of ncols values."""
    n = int(lib().qgemv_q8_1_size(int(ncols), int(batch)))
    if n < 0:
        raise ValueError("ncols must be a non-negative multiple of 32 and batch >= 1")
    return n


def q8_1_views(xq, ncols: int, batch: int):
    """(codes int8 [batch][ncols], scales fp32 [batch][ncols/32], sums int32
    [batch][ncols/32]) views of a quantized-activation buffer."""
    import torch
    _need(xq, torch.uint8, "xq")
    nq, nb = batch * ncols, batch * (ncols // QK)
    if xq.numel() < q8_1_size(ncols, batch):
        raise ValueError("xq is smaller than q8_1_size(ncols, batch)")
    q = xq[:nq].view(torch.int8).view(batch, ncols)
    d = xq[nq:nq + 4 * nb].view(torch.float32).view(batch, ncols // QK)
    s = xq[nq + 4 * nb:nq + 8 * nb].view(torch.int32).view(batch, ncols // QK)
    return q, d, s


def qquantize_q8_1(x, xq, ncols, batch, stream=None):
    """x float32 [batch][ncols] -> xq (int8 blocks of 32 with fp32 scale and
    code sum; see qgemv.h for the rounding rule)."""
    import torch
    _need(x, torch.float32, "x")
    _need(xq, torch.uint8, "xq")
    if x.numel() < batch * ncols or xq.numel() < q8_1_size(ncols, batch):
        raise ValueError("x or xq is smaller than the problem requires")
    _check(lib().qquantize_q8_1(x.data_ptr(), xq.data_ptr(), ncols, batch, _stream(x, stream)),
           "qquantize_q8_1")
    return xq


def _mmvq(fmt, W, x, y, nrows, ncols, batch, stream, pre):
    import torch
    _need(W, torch.uint8, "W")
    _need(y, torch.float32, "y")
    if pre:
        _need(x, torch.uint8, "xq")
        small = x.numel() < q8_1_size(ncols, batch)
    else:
        _need(x, torch.float32, "x")
        small = x.numel() < batch * ncols
    if W.numel() < nrows * (ncols // QK) * BLOCK_BYTES[fmt] or small or y.numel() < batch * nrows:
        raise ValueError("W, x or y is smaller than the problem requires")
    name = ("qgemv_mmvq_xq_" if pre else "qgemv_mmvq_") + fmt
    _check(getattr(lib(), name)(W.data_ptr(), x.data_ptr(), y.data_ptr(), nrows, ncols, batch,
                                _stream(W, stream)), name)
    return y


def qgemv_mmvq_q4_0(W, x, y, nrows, ncols, batch, stream=None):
    """Quantized-activation GEMV: x is quantized to int8 blocks inside the call."""
    return _mmvq("q4_0", W, x, y, nrows, ncols, batch, stream, False)


def qgemv_mmvq_q4_1(W, x, y, nrows, ncols, batch, stream=None):
    return _mmvq("q4_1", W, x, y, nrows, ncols, batch, stream, False)


def qgemv_mmvq_q8_0(W, x, y, nrows, ncols, batch, stream=None):
    return _mmvq("q8_0", W, x, y, nrows, ncols, batch, stream, False)


def qgemv_mmvq_xq_q4_0(W, xq, y, nrows, ncols, batch, stream=None):
    """Quantized-activation GEMV on activations already quantized by qquantize_q8_1."""
    return _mmvq("q4_0", W, xq, y, nrows, ncols, batch, stream, True)


def qgemv_mmvq_xq_q4_1(W, xq, y, nrows, ncols, batch, stream=None):
    return _mmvq("q4_1", W, xq, y, nrows, ncols, batch, stream, True)


def qgemv_mmvq_xq_q8_0(W, xq, y, nrows, ncols, batch, stream=None):
    return _mmvq("q8_0", W, xq, y, nrows, ncols, batch, stream, True)


def _gemv_id(fmt, W, n_expert, ids, x, x_group, y, nrows, ncols, batch, stream):
    import torch
    _need(W, torch.uint8, "W")
    _need(ids, torch.int32, "ids")
    _need(x, torch.float32, "x")
    _need(y, torch.float32, "y")
    if x_group < 1 or batch % x_group:
        raise ValueError("batch must be a multiple of x_group")
    if (W.numel() < n_expert * nrows * (ncols // QK) * BLOCK_BYTES[fmt] or ids.numel() < batch
            or x.numel() < batch // x_group * ncols or y.numel() < batch * nrows):
        raise ValueError("W, ids, x or y is smaller than the problem requires")
    name = "qgemv_id_" + fmt
    _check(getattr(lib(), name)(W.data_ptr(), n_expert, ids.data_ptr(), x.data_ptr(), x_group, y.data_ptr(),
                                nrows, ncols, batch, _stream(W, stream)), name)
    return y


def qgemv_id_q4_0(W, n_expert, ids, x, y, nrows, ncols, batch, x_group=1, stream=None):
    """Expert-selected GEMV: y[b] = W[ids[b]] . x[b // x_group] (W: n_expert matrices)."""
    return _gemv_id("q4_0", W, n_expert, ids, x, x_group, y, nrows, ncols, batch, stream)


def qgemv_id_q4_1(W, n_expert, ids, x, y, nrows, ncols, batch, x_group=1, stream=None):
    return _gemv_id("q4_1", W, n_expert, ids, x, x_group, y, nrows, ncols, batch, stream)


def qgemv_id_q8_0(W, n_expert, ids, x, y, nrows, ncols, batch, x_group=1, stream=None):
    return _gemv_id("q8_0", W, n_expert, ids, x, x_group, y, nrows, ncols, batch, stream)


def qgemv_sync_check():
    _check(lib().qgemv_sync_check(), "qgemv_sync_check")


def qgemv_version() -> int:
    return int(lib().qgemv_version())


def qgemv_shutdown() -> None:
    lib().qgemv_shutdown()


def qgemv_set_option(option: int, value: int) -> None:
    """Process-wide launch option; see qgemv.h (OPT_WEIGHTS_STATIC: the GEMV
    may start copying W before the preceding kernel of its stream finished;
    OPT_WAIT_PROBES: how long a GEMV waits for a weight copy before giving up;
    OPT_TEST_WITHHOLD_COPY: the next GEMV withholds a copy, for testing)."""
    _check(lib().qgemv_set_option(int(option), int(value)), "qgemv_set_option")
