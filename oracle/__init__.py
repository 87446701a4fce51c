"""CPU oracle for the block-quantized weight path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, the smoke check in ``__graft_entry__`` and the CPU-baseline leg
of ``bench.py`` may import this package.  The product library
(``block_quantized_weight_qgemv_gb300``) never imports, links or calls it, and
the two share no code: this package wraps ``oracle.c`` (plain C99, fp64
accumulation, bit-level fp16 / bf16 conversion) through ctypes.

What each function computes, and which page passage it follows, is stated in
``oracle.c``.  In short (the "llama_cpp 0.12.1 -> 0.12.2" diff of ggml-cuda.cu,
hunks ``dequantize_block_q4_0``, ``dequantize_block_q4_1``,
``dequantize_block_q8_0_f16`` and the to-fp16 / to-fp32 dispatch):

* ``dequant``     -- Q4_0 ``d*(q-8)``, Q4_1 ``d*q+m``, Q8_0 ``d*q`` to fp32, or to
                     fp16 by round-to-nearest-even of that fp32 value;
* ``gemv``        -- ``y[b][r] = sum_k w[r][k] * x[b][k]`` in double, rounded once;
* ``gemm``        -- ``Y[m][n] = sum_k w[n][k] * bf16(X[m][k])`` in double, rounded once;
* ``gemv_id``     -- the GEMV with output column b on expert matrix ids[b] of
                     a stack of n_expert matrices and activation row
                     b // x_group (a reading: the pages name MUL_MAT_ID
                     without printing it);
* ``quantize_q8_1`` -- activations to int8 blocks of 32 (``d = amax/127``,
                     ``q = clamp(rne(x/d), -127, 127)``, ``s = sum q``): a reading,
                     since the pages name the q8_1 conversion but print no layout;
* ``gemv_q8_1``   -- the GEMV with x replaced by ``d*q``, in double, rounded once.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(exhaustive fp16 decode against numpy, hand-built blocks under
``tests/golden/``, closed forms, brute force on tiny inputs).  Agreement with
ggml's own kernels cannot be checked (no ggml binary or printed output exists
to compare against); that cross-implementation parity is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

FMT = {"q4_0": 0, "q4_1": 1, "q8_0": 2}
BLOCK_BYTES = {"q4_0": 18, "q4_1": 20, "q8_0": 34}
QK = 32

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no FMA contraction, OpenMP if available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # QORACLE_LIB lets the mutation test load a deliberately broken build of
        # oracle.c (compiled into a temporary directory) in a child process.
        lib = ctypes.CDLL(os.environ.get("QORACLE_LIB") or build())
        i64, i32 = ctypes.c_int64, ctypes.c_int
        p = ctypes.c_void_p
        lib.oracle_fp16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_fp16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_fp16.restype = ctypes.c_uint16
        lib.oracle_block_bytes.argtypes = [i32]
        lib.oracle_block_bytes.restype = i32
        for name in ("oracle_fp16_to_f32_array", "oracle_f32_to_fp16_array",
                     "oracle_bf16_to_f32_array"):
            getattr(lib, name).argtypes = [p, p, i64]
            getattr(lib, name).restype = None
        lib.oracle_dequant.argtypes = [i32, p, i64, i64, i32, p]
        lib.oracle_dequant.restype = i32
        lib.oracle_gemv.argtypes = [i32, p, p, p, i64, i64, i64, p]
        lib.oracle_gemv.restype = i32
        lib.oracle_gemv_rows.argtypes = [i32, p, p, i64, i64, i64, p, i64, p, p]
        lib.oracle_gemv_rows.restype = i32
        lib.oracle_gemm.argtypes = [i32, p, p, p, i64, i64, i64, p]
        lib.oracle_gemm.restype = i32
        lib.oracle_gemm_entries.argtypes = [i32, p, p, i64, i64, i64, p, p, i64, p, p]
        lib.oracle_gemm_entries.restype = i32
        lib.oracle_gemv_id.argtypes = [i32, p, i64, p, p, i64, p, i64, i64, i64, p]
        lib.oracle_gemv_id.restype = i32
        lib.oracle_quantize_q8_1.argtypes = [p, i64, i64, p, p, p]
        lib.oracle_quantize_q8_1.restype = i32
        lib.oracle_gemv_q8_1.argtypes = [i32, p, p, p, p, i64, i64, i64, p]
        lib.oracle_gemv_q8_1.restype = i32
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def fp16_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().oracle_fp16_to_f32_array(_ptr(h), _ptr(out), h.size)
    return out


def f32_to_fp16(f) -> np.ndarray:
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().oracle_f32_to_fp16_array(_ptr(f), _ptr(out), f.size)
    return out


def bf16_to_f32(b) -> np.ndarray:
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float32)
    _load().oracle_bf16_to_f32_array(_ptr(b), _ptr(out), b.size)
    return out


def _check_w(fmt: str, W: np.ndarray, nrows: int, ncols: int) -> np.ndarray:
    if fmt not in FMT:
        raise ValueError("unknown format %r" % fmt)
    if ncols % QK:
        raise ValueError("ncols must be a multiple of 32")
    W = _c(W, np.uint8).reshape(-1)
    need = nrows * (ncols // QK) * BLOCK_BYTES[fmt]
    if W.size < need:
        raise ValueError("W holds %d bytes, need %d" % (W.size, need))
    return W


def dequant(fmt: str, W, nrows: int, ncols: int, out: str = "f32") -> np.ndarray:
    """[nrows][ncols] fp32 (out='f32') or fp16 bit patterns as uint16 (out='f16')."""
    W = _check_w(fmt, W, nrows, ncols)
    f16 = out == "f16"
    res = np.empty((nrows, ncols), np.uint16 if f16 else np.float32)
    rc = _load().oracle_dequant(FMT[fmt], _ptr(W), nrows, ncols, int(f16), _ptr(res))
    if rc:
        raise ValueError("oracle_dequant rejected its arguments")
    return res


def gemv(fmt: str, W, x, nrows: int, ncols: int, batch: int):
    """Returns (y [batch][nrows] fp32, absdot [batch][nrows] float64 = sum_k |w x|)."""
    W = _check_w(fmt, W, nrows, ncols)
    x = _c(x, np.float32).reshape(-1)
    if x.size < batch * ncols:
        raise ValueError("x too small")
    y = np.empty((batch, nrows), np.float32)
    ab = np.empty((batch, nrows), np.float64)
    rc = _load().oracle_gemv(FMT[fmt], _ptr(W), _ptr(x), _ptr(y), nrows, ncols, batch, _ptr(ab))
    if rc:
        raise ValueError("oracle_gemv rejected its arguments")
    return y, ab


def gemv_rows(fmt: str, W, x, nrows: int, ncols: int, batch: int, rows):
    """GEMV on a subset of rows: returns (y [batch][len(rows)], absdot likewise)."""
    W = _check_w(fmt, W, nrows, ncols)
    x = _c(x, np.float32).reshape(-1)
    rows = _c(rows, np.int64).reshape(-1)
    y = np.empty((batch, rows.size), np.float32)
    ab = np.empty((batch, rows.size), np.float64)
    rc = _load().oracle_gemv_rows(FMT[fmt], _ptr(W), _ptr(x), nrows, ncols, batch,
                                  _ptr(rows), rows.size, _ptr(y), _ptr(ab))
    if rc:
        raise ValueError("oracle_gemv_rows rejected its arguments")
    return y, ab


def gemm(fmt: str, W, X_bf16, nrows: int, ncols: int, mrows: int):
    """Returns (Y [mrows][nrows] fp32, absdot [mrows][nrows] float64)."""
    W = _check_w(fmt, W, nrows, ncols)
    X = _c(X_bf16, np.uint16).reshape(-1)
    if X.size < mrows * ncols:
        raise ValueError("X too small")
    Y = np.empty((mrows, nrows), np.float32)
    ab = np.empty((mrows, nrows), np.float64)
    rc = _load().oracle_gemm(FMT[fmt], _ptr(W), _ptr(X), _ptr(Y), nrows, ncols, mrows, _ptr(ab))
    if rc:
        raise ValueError("oracle_gemm rejected its arguments")
    return Y, ab


def gemm_entries(fmt: str, W, X_bf16, nrows: int, ncols: int, mrows: int, mi, ni):
    """GEMM on chosen entries: returns (Y[mi[i]][ni[i]] fp32, absdot float64)."""
    W = _check_w(fmt, W, nrows, ncols)
    X = _c(X_bf16, np.uint16).reshape(-1)
    mi = _c(mi, np.int64).reshape(-1)
    ni = _c(ni, np.int64).reshape(-1)
    if mi.size != ni.size:
        raise ValueError("mi and ni differ in length")
    out = np.empty(mi.size, np.float32)
    ab = np.empty(mi.size, np.float64)
    rc = _load().oracle_gemm_entries(FMT[fmt], _ptr(W), _ptr(X), nrows, ncols, mrows,
                                     _ptr(mi), _ptr(ni), mi.size, _ptr(out), _ptr(ab))
    if rc:
        raise ValueError("oracle_gemm_entries rejected its arguments")
    return out, ab


def quantize_q8_1(x, ncols: int, batch: int):
    """Quantized activations: returns (q [batch][ncols] int8, d [batch][ncols/32]
    fp32, s [batch][ncols/32] int32), the reading stated in oracle.c."""
    if ncols % QK:
        raise ValueError("ncols must be a multiple of 32")
    x = _c(x, np.float32).reshape(-1)
    if x.size < batch * ncols:
        raise ValueError("x too small")
    q = np.empty((batch, ncols), np.int8)
    d = np.empty((batch, ncols // QK), np.float32)
    s = np.empty((batch, ncols // QK), np.int32)
    rc = _load().oracle_quantize_q8_1(_ptr(x), ncols, batch, _ptr(q), _ptr(d), _ptr(s))
    if rc:
        raise ValueError("oracle_quantize_q8_1 rejected its arguments")
    return q, d, s


def gemv_q8_1(fmt: str, W, q, d, nrows: int, ncols: int, batch: int):
    """GEMV on quantized activations xhat = d*q: returns (y [batch][nrows] fp32,
    absdot [batch][nrows] float64 = sum_k |w xhat|)."""
    W = _check_w(fmt, W, nrows, ncols)
    q = _c(q, np.int8).reshape(-1)
    d = _c(d, np.float32).reshape(-1)
    if q.size < batch * ncols or d.size < batch * (ncols // QK):
        raise ValueError("q or d too small")
    y = np.empty((batch, nrows), np.float32)
    ab = np.empty((batch, nrows), np.float64)
    rc = _load().oracle_gemv_q8_1(FMT[fmt], _ptr(W), _ptr(q), _ptr(d), _ptr(y), nrows, ncols,
                                  batch, _ptr(ab))
    if rc:
        raise ValueError("oracle_gemv_q8_1 rejected its arguments")
    return y, ab


def gemv_id(fmt: str, W, n_expert: int, ids, x, nrows: int, ncols: int, batch: int, x_group: int = 1):
    """Expert-selected GEMV: returns (y [batch][nrows] fp32, absdot float64).
    x holds batch // x_group activation rows."""
    W = _check_w(fmt, W, nrows * n_expert, ncols)
    ids = _c(ids, np.int32).reshape(-1)
    x = _c(x, np.float32).reshape(-1)
    if x_group < 1 or batch % x_group:
        raise ValueError("batch must be a multiple of x_group")
    if ids.size < batch or x.size < batch // x_group * ncols:
        raise ValueError("ids or x too small")
    y = np.empty((batch, nrows), np.float32)
    ab = np.empty((batch, nrows), np.float64)
    rc = _load().oracle_gemv_id(FMT[fmt], _ptr(W), n_expert, _ptr(ids), _ptr(x), x_group, _ptr(y), nrows,
                                ncols, batch, _ptr(ab))
    if rc:
        raise ValueError("oracle_gemv_id rejected its arguments")
    return y, ab
