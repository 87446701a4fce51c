"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and
the benchmark.

This module only draws random numbers and packs them into the ggml block byte
layouts; it holds none of the method's arithmetic (no dequantization, no dot
products).  Layouts: Q4_0 ``[d:fp16][qs:16 bytes]`` (18 B), Q4_1
``[d:fp16][m:fp16][qs:16 bytes]`` (20 B), Q8_0 ``[d:fp16][qs:32 x int8]`` (34 B);
a row of ``ncols`` weights is ``ncols/32`` consecutive blocks, rows consecutive.

Distributions (the workload recipe):

* Q4_0: ``d = fp16(U[1e-3, 1e-2])``, the 16 ``qs`` bytes ``U{0..255}``;
* Q4_1: ``d = fp16(U[1e-3, 1e-2])``, ``m = fp16(U[-0.08, 0])``, bytes ``U{0..255}``;
* Q8_0: ``d = fp16(U[1e-4, 1e-3])``, ``qs`` int8 ``U{-127..127}``;
* x: fp32 ``N(0, 1)``;  X (prefill activations): ``N(0, 1)`` rounded to bf16 (RNE).

Every generator takes an explicit seed (numpy ``PCG64``).
"""
from __future__ import annotations

import numpy as np

QK = 32
BLOCK_BYTES = {"q4_0": 18, "q4_1": 20, "q8_0": 34}

D_RANGE = {"q4_0": (1e-3, 1e-2), "q4_1": (1e-3, 1e-2), "q8_0": (1e-4, 1e-3)}
M_RANGE_Q4_1 = (-0.08, 0.0)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def pack_blocks(fmt: str, d: np.ndarray, qs: np.ndarray, m: np.ndarray | None = None) -> np.ndarray:
    """Pack per-block fields into the block byte layout.

    d, m: float16 arrays of shape [nblocks]; qs: uint8 [nblocks, 16] (Q4_*) or
    int8/uint8 [nblocks, 32] (Q8_0).  Returns uint8 [nblocks * block_bytes].
    """
    d = np.ascontiguousarray(d, np.float16).reshape(-1)
    nblk = d.size
    bb = BLOCK_BYTES[fmt]
    out = np.empty((nblk, bb), np.uint8)
    out[:, 0:2] = d.view(np.uint8).reshape(nblk, 2)
    if fmt == "q4_1":
        if m is None:
            raise ValueError("Q4_1 needs m")
        out[:, 2:4] = np.ascontiguousarray(m, np.float16).reshape(-1).view(np.uint8).reshape(nblk, 2)
        out[:, 4:20] = np.ascontiguousarray(qs).view(np.uint8).reshape(nblk, 16)
    elif fmt == "q4_0":
        out[:, 2:18] = np.ascontiguousarray(qs).view(np.uint8).reshape(nblk, 16)
    elif fmt == "q8_0":
        out[:, 2:34] = np.ascontiguousarray(qs).view(np.uint8).reshape(nblk, 32)
    else:
        raise ValueError(fmt)
    return out.reshape(-1)


def make_weights(fmt: str, nrows: int, ncols: int, seed: int) -> np.ndarray:
    """Random blocks for an nrows x ncols weight matrix; uint8 [nrows * ncols/32 * bb]."""
    if ncols % QK:
        raise ValueError("ncols must be a multiple of 32")
    g = rng(seed)
    nblk = nrows * (ncols // QK)
    lo, hi = D_RANGE[fmt]
    d = g.uniform(lo, hi, nblk).astype(np.float16)
    if fmt == "q8_0":
        qs = g.integers(-127, 128, (nblk, 32), dtype=np.int8)
        return pack_blocks(fmt, d, qs)
    qs = g.integers(0, 256, (nblk, 16), dtype=np.uint8)
    m = None
    if fmt == "q4_1":
        m = g.uniform(M_RANGE_Q4_1[0], M_RANGE_Q4_1[1], nblk).astype(np.float16)
    return pack_blocks(fmt, d, qs, m)


def make_x(batch: int, ncols: int, seed: int) -> np.ndarray:
    """fp32 N(0,1) activations [batch][ncols]."""
    return rng(seed).standard_normal((batch, ncols), dtype=np.float32)


def round_f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (nearest, ties to even); uint16 bit patterns.

    Input-generation helper only: used to draw bf16 activations."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    nan = np.isnan(np.asarray(a, np.float32))
    r = np.where(nan, (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def make_X_bf16(mrows: int, ncols: int, seed: int) -> np.ndarray:
    """bf16 N(0,1) prefill activations [mrows][ncols] as uint16 bit patterns."""
    return round_f32_to_bf16_bits(rng(seed).standard_normal((mrows, ncols), dtype=np.float32))
