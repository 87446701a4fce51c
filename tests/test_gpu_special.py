"""GPU parity on the inputs the random workloads never produce, through the C ABI.

Each case runs the kernel the dispatch picks for its shape (ncols a multiple of
2048: the stream-K tensor-core GEMV; 4096 x 14336 at batch 8: the cluster-split
tensor-core GEMV, whose staged x does not fit one CTA) and compares every
element with the oracle at the stated bound
|y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-6.

Weights (block formulas of the dequantize_block_q4_0 / _q4_1 / _q8_0_f16 hunks
of the "llama_cpp 0.12.1 -> 0.12.2" ggml-cuda.cu diff):
  - scales d = +0, -0 and 2^-24 (the smallest fp16 subnormal) in scattered blocks;
  - Q8_0 codes -128 (outside the workloads' -127..127 draw);
  - whole rows of zero weights with nonzero d (Q4_0 nibbles all 8, Q8_0 codes 0,
    Q4_1 d = m = 0), whose exact product is 0: the bound is then 1e-6;
  - a column k* whose weight is zero in every third row.
Activations per batch column: N(0,1); all zero; one-hot; N(0,1) with x[k*] =
1e11 (the rows whose weight at k* is zero must still get the N(0,1) part right);
N(0,1) with a few values near 1e-30 (a dynamic range far beyond fp16's inside
one block); N(0,1) scaled by 1e-30 and by 1e30.
The output sits between guard bands of 256 floats on each side that must come
back untouched.
"""
import numpy as np
import pytest

import qsynth
from gpu_util import assert_within_bound, qlib, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

FMTS = ["q4_0", "q4_1", "q8_0"]
GUARD = 256
SENTINEL = -7.25


def special_weights(fmt, nrows, ncols, seed, kstar):
    g = qsynth.rng(seed)
    nb = ncols // 32
    nblk = nrows * nb
    lo, hi = qsynth.D_RANGE[fmt]
    d = g.uniform(lo, hi, nblk).astype(np.float16)
    d[::7] = np.float16(0.0)
    d[1::7] = np.float16(-0.0)
    d[2::11] = np.float16(2.0 ** -24)
    kb, kj = kstar // 32, kstar % 32
    zero_rows = list(range(1, nrows, 3))
    blank_row = nrows // 2                       # every weight of this row is 0
    m = None
    if fmt == "q8_0":
        qs = g.integers(-127, 128, (nblk, 32), dtype=np.int8)
        qs[::5, 3] = -128
        qs[3::13, :] = -128
        for r in zero_rows:
            qs[r * nb + kb, kj] = 0
        qs[blank_row * nb:(blank_row + 1) * nb, :] = 0
        d[blank_row * nb:(blank_row + 1) * nb] = np.float16(3e-4)
    else:
        qs = g.integers(0, 256, (nblk, 16), dtype=np.uint8)
        if fmt == "q4_1":
            m = g.uniform(qsynth.M_RANGE_Q4_1[0], qsynth.M_RANGE_Q4_1[1], nblk).astype(np.float16)
            m[5::9] = np.float16(-0.0)
        for r in zero_rows:
            i = r * nb + kb
            if fmt == "q4_0":                    # nibble 8 -> weight 0
                b = kj % 16
                qs[i, b] = (qs[i, b] & 0xF0) | 0x08 if kj < 16 else (qs[i, b] & 0x0F) | 0x80
            else:                                # Q4_1: zero the whole block
                d[i] = np.float16(0.0)
                m[i] = np.float16(0.0)
        if fmt == "q4_0":
            qs[blank_row * nb:(blank_row + 1) * nb, :] = 0x88
            d[blank_row * nb:(blank_row + 1) * nb] = np.float16(5e-3)
        else:
            d[blank_row * nb:(blank_row + 1) * nb] = np.float16(0.0)
            m[blank_row * nb:(blank_row + 1) * nb] = np.float16(0.0)
    return qsynth.pack_blocks(fmt, d, qs, m), blank_row


def special_x(batch, ncols, seed, kstar):
    g = qsynth.rng(seed)
    kinds = []
    x = np.zeros((batch, ncols), np.float32)
    for n in range(batch):
        kind = n % 7
        base = g.standard_normal(ncols, dtype=np.float32)
        if kind == 0:
            x[n] = base
        elif kind == 1:
            x[n] = 0.0
        elif kind == 2:
            x[n, (kstar * 7 + 5) % ncols] = 1.0
        elif kind == 3:
            x[n] = base
            x[n, kstar] = 1e11
        elif kind == 4:
            x[n] = base
            x[n, g.integers(0, ncols, 9)] = np.float32(1e-30)
        elif kind == 5:
            x[n] = base * np.float32(1e-30)
        else:
            x[n] = base * np.float32(1e30)
        kinds.append(kind)
    return x, kinds


def run_guarded(q, torch, fn, args, nout):
    buf = torch.full((2 * GUARD + nout,), SENTINEL, dtype=torch.float32, device="cuda")
    out = buf[GUARD:GUARD + nout]
    fn(*args(out))
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    b = buf.cpu().numpy()
    assert np.all(b[:GUARD] == SENTINEL) and np.all(b[GUARD + nout:] == SENTINEL), "guard band overwritten"
    return b[GUARD:GUARD + nout]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape,batch", [((77, 2048), 1), ((77, 2048), 3), ((300, 4096), 7),
                                         ((4096, 14336), 1), ((4096, 14336), 8)])
def test_gemv_special_values(oracle_mod, fmt, shape, batch):
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = shape
    kstar = ncols // 2 + 37
    Wn, blank = special_weights(fmt, nrows, ncols, 40 + nrows, kstar)
    xn, kinds = special_x(batch, ncols, 41, kstar)
    if batch == 1:
        xn[0, kstar] = 1e11                      # the large-range case at batch 1 too
    W, x = to_dev(Wn, torch), to_dev(xn, torch)
    got = run_guarded(q, torch, getattr(q, "qgemv_" + fmt),
                      lambda out: (W, x, out.view(batch, nrows), nrows, ncols, batch), batch * nrows)
    got = got.reshape(batch, nrows)
    ref, ab = oracle_mod.gemv(fmt, Wn, xn, nrows, ncols, batch)
    assert_within_bound(got, ref, ab, "%s %dx%d b%d special" % (fmt, nrows, ncols, batch))
    # exact zeros where the product is exactly zero
    assert np.all(got[:, blank] == 0.0)
    for n, kind in enumerate(kinds):
        if kind == 1:
            assert np.all(got[n] == 0.0)


@pytest.mark.parametrize("batch", [1, 2, 3, 8])
@pytest.mark.parametrize("spike", [1e3, 1e6, 3e7])
def test_gemv_q4_1_cancelling_zero_weights(oracle_mod, batch, spike):
    """Q4_1 weights that are exactly zero through d*q + m = 0 with d, m != 0
    (d = 2^-7, m = -8 * 2^-7, q = 8) at a column carrying a large value: the
    products d * sum(q x) and m * sum(x) cancel, and the result must still be
    the N(0,1) part within the bound."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = 300, 4096
    nb = ncols // 32
    g = np.random.default_rng(int(spike) % 1000 + batch)
    d = np.full(nrows * nb, np.float16(2.0 ** -7))
    m = np.full(nrows * nb, np.float16(-8 * 2.0 ** -7))
    qs = g.integers(0, 256, (nrows * nb, 16), dtype=np.uint8)
    k = 1234
    kb, kj = k // 32, k % 32
    for r in range(nrows):
        i, b = r * nb + kb, kj % 16
        qs[i, b] = (qs[i, b] & 0xF0) | 0x08 if kj < 16 else (qs[i, b] & 0x0F) | 0x80
    Wn = qsynth.pack_blocks("q4_1", d, qs, m)
    xn = qsynth.make_x(batch, ncols, seed=7).copy()
    xn[:, k] = spike
    W, x = to_dev(Wn, torch), to_dev(xn, torch)
    got = run_guarded(q, torch, q.qgemv_q4_1, lambda out: (W, x, out.view(batch, nrows), nrows, ncols, batch),
                      batch * nrows).reshape(batch, nrows)
    ref, ab = oracle_mod.gemv("q4_1", Wn, xn, nrows, ncols, batch)
    assert_within_bound(got, ref, ab, "q4_1 cancelling zero weights, spike %g, b%d" % (spike, batch))


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_deterministic_special(fmt):
    """Bitwise equal results on repeated calls, including the exact fallback
    for chunks whose dynamic range exceeds fp16's."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, batch = 4096, 14336, 5
    kstar = 7000
    Wn, _ = special_weights(fmt, nrows, ncols, 3, kstar)
    xn, _ = special_x(batch, ncols, 4, kstar)
    W, x = to_dev(Wn, torch), to_dev(xn, torch)
    outs = []
    for _ in range(3):
        y = torch.empty(batch, nrows, dtype=torch.float32, device="cuda")
        getattr(q, "qgemv_" + fmt)(W, x, y, nrows, ncols, batch)
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy().view(np.uint32))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_gemv_wait_timeout_reported_and_recovered(oracle_mod):
    """A GEMV whose first weight copy is withheld (a wait nothing completes)
    gives up after the configured probes, reports QGEMV_ERR_TIMEOUT through
    qgemv_sync_check, and the next call is correct."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = 512, 4096
    Wn = qsynth.make_weights("q4_0", nrows, ncols, 77)
    xn = qsynth.make_x(1, ncols, 78)
    W, x = to_dev(Wn, torch), to_dev(xn, torch)
    y = torch.empty(1, nrows, dtype=torch.float32, device="cuda")
    q.qgemv_set_option(q.OPT_WAIT_PROBES, 2000)
    try:
        q.qgemv_set_option(q.OPT_TEST_WITHHOLD_COPY, 1)
        q.qgemv_q4_0(W, x, y, nrows, ncols, 1)
        with pytest.raises(q.QgemvError) as e:
            q.qgemv_sync_check()
        assert e.value.status == 8
    finally:
        q.qgemv_set_option(q.OPT_WAIT_PROBES, 1 << 20)
        q.qgemv_set_option(q.OPT_TEST_WITHHOLD_COPY, 0)
    for _ in range(2):
        y.fill_(float("nan"))
        q.qgemv_q4_0(W, x, y, nrows, ncols, 1)
        torch.cuda.synchronize()
        q.qgemv_sync_check()
        ref, ab = oracle_mod.gemv("q4_0", Wn, xn, nrows, ncols, 1)
        assert_within_bound(y.cpu().numpy(), ref, ab, "after timeout")



def special_X(m, ncols, seed, kstar):
    """Token rows for the prefill (bf16): N(0,1); zero; one-hot; N(0,1) x 1e-30;
    N(0,1) x 1e30; N(0,1) with a few values near 1e-30; N(0,1) x 3e4 with
    +-65504 and +-1e5 entries (beyond fp16's range before the row scaling)."""
    g = qsynth.rng(seed)
    X = np.zeros((m, ncols), np.float32)
    for i in range(m):
        kind = i % 7
        base = g.standard_normal(ncols, dtype=np.float32)
        if kind == 0:
            X[i] = base
        elif kind == 1:
            X[i] = 0.0
        elif kind == 2:
            X[i, (kstar * 5 + 3) % ncols] = 1.0
        elif kind == 3:
            X[i] = base * np.float32(1e-30)
        elif kind == 4:
            X[i] = base * np.float32(1e30)
        elif kind == 5:
            X[i] = base
            X[i, g.integers(0, ncols, 9)] = np.float32(1e-30)
        else:
            X[i] = base * np.float32(3e4)
            X[i, kstar] = 65504.0
            X[i, (kstar + 1) % ncols] = -1e5
    return qsynth.round_f32_to_bf16_bits(X)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(77, 2048, 9), (300, 1024, 130)])
def test_gemm_special_values(oracle_mod, fmt, shape):
    """The tensor-core prefill on the special weights and on token rows that
    span the bf16 range, with guard bands around Y."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, m = shape
    kstar = ncols // 2 + 37
    Wn, blank = special_weights(fmt, nrows, ncols, 60 + nrows, kstar)
    Xn = special_X(m, ncols, 61, kstar)
    W = to_dev(Wn, torch)
    X = torch.from_numpy(Xn.view(np.int16)).cuda().view(torch.bfloat16)
    got = run_guarded(q, torch, getattr(q, "qgemm_" + fmt),
                      lambda out: (W, X, out.view(m, nrows), nrows, ncols, m), m * nrows)
    got = got.reshape(m, nrows)
    ref, ab = oracle_mod.gemm(fmt, Wn, Xn, nrows, ncols, m)
    assert_within_bound(got, ref, ab, "%s prefill %s special" % (fmt, shape))
    assert np.all(got[:, blank] == 0.0)
    assert np.all(got[1::7] == 0.0)


def emulate_row_f16(xrow):
    """The prefill's documented operand rounding of one token row: scaled by
    the power of two that puts its largest magnitude in [2^14, 2^15), rounded
    to fp16 (values below fp16's range flush to zero or to subnormals), then
    scaled back -- so nonzero values more than 2^28 below the row's largest
    lose bits or vanish."""
    x = np.asarray(xrow, np.float64)
    amax = np.max(np.abs(x))
    if amax == 0 or not np.isfinite(amax):
        return x.astype(np.float32)
    e = 14 - int(np.floor(np.log2(amax)))
    scaled = (x * 2.0 ** e).astype(np.float16).astype(np.float64)
    return (scaled * 2.0 ** -e).astype(np.float32)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_domain_limit(oracle_mod, fmt):
    """Token rows outside the prefill's stated domain: a 1e30 spike at a column
    k* (where every third weight row is zero) beside N(0,1) values 2^99 below
    it.  The result must equal the product of the rows as the documented
    rounding leaves them (the N(0,1) part lost), within the GEMV bound of
    that product -- in particular exactly 0 on the rows whose weight at k* is
    zero; in-domain rows are unaffected."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, m = 77, 1024, 6
    kstar = ncols // 2 + 37
    Wn, _ = special_weights(fmt, nrows, ncols, 90, kstar)
    g = np.random.default_rng(91)
    X = g.standard_normal((m, ncols)).astype(np.float32)
    X[::2, kstar] = 1e30                      # rows 0, 2, 4 out of the domain
    Xb = qsynth.round_f32_to_bf16_bits(X)
    Xf = (Xb.astype(np.uint32) << 16).view(np.float32)
    W = to_dev(Wn, torch)
    Xd = torch.from_numpy(Xb.view(np.int16)).cuda().view(torch.bfloat16)
    got = run_guarded(q, torch, getattr(q, "qgemm_" + fmt),
                      lambda out: (W, Xd, out.view(m, nrows), nrows, ncols, m), m * nrows).reshape(m, nrows)
    Xe = np.stack([emulate_row_f16(Xf[i]) for i in range(m)])
    assert np.count_nonzero(Xe[0]) == 1       # the spike alone survives the rounding
    ref, ab = oracle_mod.gemv(fmt, Wn, Xe, nrows, ncols, m)
    assert_within_bound(got, ref, ab, "%s prefill outside the domain" % fmt)
    zero_rows = list(range(1, nrows, 3))
    assert np.all(got[0, zero_rows] == 0.0)
