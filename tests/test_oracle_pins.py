"""Pins of the CPU oracle against facts that do not come from the oracle itself.

* fp16 decode: all 65,536 bit patterns against numpy's float16 (an independent
  implementation);
* fp32 -> fp16 round-to-nearest-even: random bit patterns plus every fp16
  boundary, midpoint and neighbour against numpy's ``astype(float16)``;
* bf16 decode: all 65,536 patterns against torch's bfloat16;
* dequantization: hand-built blocks with closed-form values
  (``tests/golden/blocks.txt``), a one-hot sweep of every nibble / byte
  position, quantize-then-dequantize of exactly representable values, and the
  row / block stride on multi-row matrices with per-block closed forms;
* GEMV / GEMM: one-hot activations (each output equals one weight), brute
  force in float64 with numpy on tiny matrices, row sums against closed forms,
  batch independence and the sampled-entry forms;
* quantized activations (q8_1): hand-built blocks with closed-form codes
  (ties to even), exact multiples of a scale, zero / non-finite / subnormal
  scale blocks, numpy's round-half-even as an independent rounding routine,
  the GEMV on exactly representable x against the plain GEMV, an integer-dot
  form from a numpy decode of the raw bytes, and the stated error bound.

Formulas: "llama_cpp 0.12.1 -> 0.12.2" diff of ggml-cuda.cu, hunks adding
dequantize_block_q4_0 / dequantize_block_q4_1 / dequantize_block_q8_0_f16;
the format statement (Q4_0 w = d*(q-8), Q4_1 w = d*q + m, Q8_0 w = d*q).
"""
import numpy as np
import pytest

import qsynth
from golden_io import load_blocks

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bits32(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


# ---------------------------------------------------------------- fp16 / bf16

def test_fp16_decode_exhaustive(oracle_mod):
    h = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.fp16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(bits32(got)[~nan], bits32(ref)[~nan])


def _fp16_boundary_values():
    h = np.arange(0, 0x7C00, dtype=np.uint16)            # all finite non-negative fp16
    v = h.view(np.float16).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2.0                           # exact ties (representable in fp32)
    vals = [v, mids, np.array([65504.0, 65519.99, 65520.0, 65536.0, 1e30, 2.0**-25, 2.0**-26, 3 * 2.0**-26])]
    out = np.concatenate(vals).astype(np.float32)
    up = np.nextafter(out, np.float32(np.inf))
    dn = np.nextafter(out, np.float32(0))
    allv = np.concatenate([out, up, dn])
    return np.concatenate([allv, -allv])


def test_f32_to_fp16_rne(oracle_mod):
    g = qsynth.rng(11)
    rnd = g.integers(0, 2**32, 1_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    f = np.concatenate([_fp16_boundary_values(), rnd,
                        np.array([np.inf, -np.inf, np.nan, 0.0, -0.0], np.float32)])
    got = oracle_mod.f32_to_fp16(f)
    ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(np.isnan(got.view(np.float16)), nan)
    bad = np.nonzero(got[~nan] != ref[~nan])[0]
    assert bad.size == 0, (f[~nan][bad[:5]], got[~nan][bad[:5]], ref[~nan][bad[:5]])


def test_bf16_decode_exhaustive(oracle_mod):
    torch = pytest.importorskip("torch")
    b = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.bf16_to_f32(b)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(bits32(got)[~nan], bits32(ref)[~nan])


# ------------------------------------------------------------ golden blocks

CASES = load_blocks()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_golden_block(oracle_mod, case):
    w = oracle_mod.dequant(case["format"], case["bytes"], 1, 32, out="f32").reshape(-1)
    assert np.array_equal(bits32(w), bits32(case["f32"])), (w, case["f32"])
    h = oracle_mod.dequant(case["format"], case["bytes"], 1, 32, out="f16").reshape(-1)
    if "f16" in case:
        assert np.array_equal(h, case["f16"]), (h, case["f16"])
    # fp16 output is the RNE rounding of the fp32 value (checked with numpy's rounding)
    assert np.array_equal(h, case["f32"].astype(np.float16).view(np.uint16))


def test_golden_fixture_matches_closed_forms():
    """The fixture text agrees with the closed forms its 'why' lines state."""
    by = {c["name"]: c for c in CASES}
    j = np.arange(16)
    assert np.array_equal(by["q4_0_ramp_d1"]["f32"], np.concatenate([j - 8, 7 - j]).astype(np.float32))
    assert np.array_equal(by["q4_1_ramp"]["f32"], np.concatenate([2 * j - 3, 27 - 2 * j]).astype(np.float32))
    jj = np.arange(32)
    assert np.array_equal(by["q8_0_quarters"]["f32"], ((8 * jj - 128) / 4).astype(np.float32))


# -------------------------------------------------- nibble / byte positions

@pytest.mark.parametrize("fmt", ["q4_0", "q4_1"])
def test_every_nibble_position(oracle_mod, fmt):
    """Setting one nibble moves exactly one element: low nibble of qs[j] ->
    element j, high nibble -> element j+16."""
    d = np.float16(0.5)
    m = np.float16(0.0)
    base = 8 if fmt == "q4_0" else 0
    blocks = []
    for pos in range(32):
        qs = np.full(16, base | (base << 4), np.uint8)
        j, hi = pos % 16, pos >= 16
        nib = base + 3
        qs[j] = (qs[j] & 0x0F) | (nib << 4) if hi else (qs[j] & 0xF0) | nib
        blocks.append(qsynth.pack_blocks(fmt, np.array([d]), qs[None], np.array([m]) if fmt == "q4_1" else None))
    W = np.concatenate(blocks)
    w = oracle_mod.dequant(fmt, W, 32, 32)
    expect = np.zeros((32, 32), np.float32)
    expect[np.arange(32), np.arange(32)] = 1.5          # 0.5 * 3
    assert np.array_equal(w, expect)


def test_q8_0_every_byte_and_sign(oracle_mod):
    d = np.float16(2.0)
    blocks = []
    for pos in range(32):
        qs = np.zeros(32, np.int8)
        qs[pos] = -128 if pos % 2 else 127
        blocks.append(qsynth.pack_blocks("q8_0", np.array([d]), qs[None]))
    w = oracle_mod.dequant("q8_0", np.concatenate(blocks), 32, 32)
    expect = np.zeros((32, 32), np.float32)
    expect[np.arange(32), np.arange(32)] = np.where(np.arange(32) % 2, -256.0, 254.0)
    assert np.array_equal(w, expect)


# ------------------------------------------------------ quantize round trip

def _roundtrip_case(fmt, seed):
    """Draw representable values v, quantize them with a test-local quantizer
    for a known scale, and return (blocks, v).  v is built from the integer
    codes with float64 arithmetic, which is exact for these magnitudes."""
    g = qsynth.rng(seed)
    nblk = 64
    e = g.integers(-12, 4, nblk)
    d = (2.0 ** e) * g.choice([1.0, 1.25, 1.5, 1.75], nblk)          # exact in fp16
    if fmt == "q8_0":
        q = g.integers(-128, 128, (nblk, 32))
        v = d[:, None] * q
        qq = np.rint(v / d[:, None]).astype(np.int64)
        return qsynth.pack_blocks(fmt, d.astype(np.float16), qq.astype(np.int8)), v
    q = g.integers(0, 16, (nblk, 32))
    if fmt == "q4_0":
        v = d[:, None] * (q - 8)
        qq = np.rint(v / d[:, None]).astype(np.int64) + 8
        m = None
    else:
        m = -(2.0 ** g.integers(-6, 2, nblk))                         # exact in fp16
        v = d[:, None] * q + m[:, None]                               # exact in fp32 (<= 24 bits span)
        qq = np.rint((v - m[:, None]) / d[:, None]).astype(np.int64)
        m = m.astype(np.float16)
    packed = (qq[:, :16] | (qq[:, 16:] << 4)).astype(np.uint8)
    return qsynth.pack_blocks(fmt, d.astype(np.float16), packed, m), v


@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q8_0"])
def test_quantize_dequantize_roundtrip(oracle_mod, fmt):
    W, v = _roundtrip_case(fmt, {"q4_0": 1, "q4_1": 2, "q8_0": 3}[fmt])
    w = oracle_mod.dequant(fmt, W, 64, 32)
    assert np.array_equal(w.astype(np.float64), v)


# ----------------------------------------------------- row / block strides

@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q8_0"])
def test_row_and_block_stride(oracle_mod, fmt):
    """3 rows x 5 blocks; block (r, b) has scale 2^-(r*5+b) and constant code,
    so element [r][32b + j] has a closed form."""
    nrows, nb = 3, 5
    idx = np.arange(nrows * nb)
    d = (2.0 ** -idx).astype(np.float16)
    if fmt == "q8_0":
        qs = np.full((idx.size, 32), 3, np.int8)
        W = qsynth.pack_blocks(fmt, d, qs)
        per = 3.0 * 2.0 ** -idx
    else:
        qs = np.full((idx.size, 16), 0xBB, np.uint8)                   # nibble 11
        m = np.zeros(idx.size, np.float16) if fmt == "q4_1" else None
        W = qsynth.pack_blocks(fmt, d, qs, m)
        per = (11 - 8 if fmt == "q4_0" else 11) * 2.0 ** -idx
    w = oracle_mod.dequant(fmt, W, nrows, nb * 32)
    expect = np.repeat(per.reshape(nrows, nb), 32, axis=1).astype(np.float32)
    assert np.array_equal(w, expect)


def test_f16_output_rounds_the_f32_value(oracle_mod):
    for fmt in ("q4_0", "q4_1", "q8_0"):
        W = qsynth.make_weights(fmt, 7, 96, seed=5)
        f32 = oracle_mod.dequant(fmt, W, 7, 96, out="f32")
        f16 = oracle_mod.dequant(fmt, W, 7, 96, out="f16")
        assert np.array_equal(f16, f32.astype(np.float16).view(np.uint16))


# --------------------------------------------------------------- GEMV / GEMM

@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q8_0"])
def test_gemv_one_hot_picks_weights(oracle_mod, fmt):
    """x = e_k (batch k) gives y[k][r] = w[r][k] exactly: pins the operand
    orientation and indexing of the contraction."""
    nrows, ncols = 5, 96
    W = qsynth.make_weights(fmt, nrows, ncols, seed=21)
    w = oracle_mod.dequant(fmt, W, nrows, ncols)
    x = np.eye(ncols, dtype=np.float32)                        # batch = ncols one-hot rows
    y, ab = oracle_mod.gemv(fmt, W, x, nrows, ncols, ncols)
    assert np.array_equal(y, w.T)
    assert np.array_equal(ab, np.abs(w.T).astype(np.float64))


@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q8_0"])
@pytest.mark.parametrize("shape", [(3, 64, 1), (5, 96, 3), (4, 256, 2)])
def test_gemv_brute_force_float64(oracle_mod, fmt, shape):
    nrows, ncols, batch = shape
    W = qsynth.make_weights(fmt, nrows, ncols, seed=31)
    x = qsynth.make_x(batch, ncols, seed=32)
    w = oracle_mod.dequant(fmt, W, nrows, ncols).astype(np.float64)
    ref = x.astype(np.float64) @ w.T                            # [batch][nrows]
    y, ab = oracle_mod.gemv(fmt, W, x, nrows, ncols, batch)
    assert y.shape == (batch, nrows)
    assert np.allclose(y, ref.astype(np.float32), rtol=1e-6, atol=1e-12)
    assert np.allclose(ab, np.abs(x.astype(np.float64)[:, None, :] * w[None]).sum(-1), rtol=1e-12)


def test_gemv_row_sums_closed_form(oracle_mod):
    """x = 1: y[r] = sum of row r's weights; ramp blocks sum to d*(sum(j-8) + sum(7-j)) = -16 d."""
    ramp = np.array([j | ((15 - j) << 4) for j in range(16)], np.uint8)
    nrows, nb = 4, 3
    d = (2.0 ** -np.arange(nrows * nb)).astype(np.float16)
    W = qsynth.pack_blocks("q4_0", d, np.tile(ramp, (nrows * nb, 1)))
    y, _ = oracle_mod.gemv("q4_0", W, np.ones((1, nb * 32), np.float32), nrows, nb * 32, 1)
    expect = (-16.0 * d.astype(np.float64).reshape(nrows, nb)).sum(1)
    assert np.array_equal(y[0].astype(np.float64), expect)


def test_gemv_batch_independent(oracle_mod):
    W = qsynth.make_weights("q4_1", 6, 128, seed=41)
    x = qsynth.make_x(4, 128, seed=42)
    y, ab = oracle_mod.gemv("q4_1", W, x, 6, 128, 4)
    for b in range(4):
        yb, abb = oracle_mod.gemv("q4_1", W, x[b:b + 1], 6, 128, 1)
        assert np.array_equal(yb[0], y[b]) and np.array_equal(abb[0], ab[b])


def test_gemv_rows_matches_full(oracle_mod):
    W = qsynth.make_weights("q8_0", 40, 64, seed=51)
    x = qsynth.make_x(3, 64, seed=52)
    y, ab = oracle_mod.gemv("q8_0", W, x, 40, 64, 3)
    rows = np.array([0, 39, 7, 7, 21])
    ys, abs_ = oracle_mod.gemv_rows("q8_0", W, x, 40, 64, 3, rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(abs_, ab[:, rows])


def test_gemm_matches_gemv_on_decoded_rows(oracle_mod):
    """Row m of the prefill matmul is the GEMV of bf16(X[m]) (decoded by torch)."""
    torch = pytest.importorskip("torch")
    nrows, ncols, mrows = 9, 128, 5
    W = qsynth.make_weights("q4_0", nrows, ncols, seed=61)
    X = qsynth.make_X_bf16(mrows, ncols, seed=62)
    Y, ab = oracle_mod.gemm("q4_0", W, X, nrows, ncols, mrows)
    xf = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).float().numpy()
    y2, ab2 = oracle_mod.gemv("q4_0", W, xf, nrows, ncols, mrows)
    assert np.array_equal(Y, y2) and np.array_equal(ab, ab2)
    w = oracle_mod.dequant("q4_0", W, nrows, ncols).astype(np.float64)
    assert np.allclose(Y, (xf.astype(np.float64) @ w.T).astype(np.float32), rtol=1e-6, atol=1e-12)


def test_gemm_entries_matches_full(oracle_mod):
    W = qsynth.make_weights("q4_1", 12, 64, seed=71)
    X = qsynth.make_X_bf16(6, 64, seed=72)
    Y, ab = oracle_mod.gemm("q4_1", W, X, 12, 64, 6)
    mi = np.array([0, 5, 3, 3])
    ni = np.array([11, 0, 4, 5])
    v, a = oracle_mod.gemm_entries("q4_1", W, X, 12, 64, 6, mi, ni)
    assert np.array_equal(v, Y[mi, ni]) and np.array_equal(a, ab[mi, ni])


def test_bad_arguments_rejected(oracle_mod):
    W = qsynth.make_weights("q4_0", 2, 64, seed=1)
    with pytest.raises(ValueError):
        oracle_mod.dequant("q4_0", W, 2, 63)
    with pytest.raises(ValueError):
        oracle_mod.dequant("q5_0", W, 2, 64)
    with pytest.raises(ValueError):
        oracle_mod.gemv_rows("q4_0", W, np.zeros(64, np.float32), 2, 64, 1, [2])


# ----------------------------------------------- quantized activations (q8_1)
#
# The pages name the int8 activation blocks of the mul_mat_vec_q family
# (convert_src1_to_q8_1 in ggml_cuda_op_mul_mat, the __dp4a note beside
# MIN_CC_DP4A) without printing their layout; the reading pinned here is
# d = amax/127, q = clamp(rne(x/d), -127, 127), s = sum(q).

def _q8_1_hand_block():
    """One block with amax = 127 (so d = 1 exactly) and closed-form codes:
    ties go to the even neighbour, everything else to the nearest integer."""
    vals = [127.0, -127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5,
            3.4999998, 3.5000002, 126.5, -126.5, 0.0, -0.0, 100.25, -100.75,
            0.49999997, 5.5, 6.5, -5.5, -6.5, 64.0, -64.0, 7.0,
            1e-30, -1e-30, 99.5, 98.5, -98.5, 12.75, -12.25, 42.0]
    codes = [127, -127, 0, 2, 2, 0, -2, -2,
             3, 4, 126, -126, 0, 0, 100, -101,
             0, 6, 6, -6, -6, 64, -64, 7,
             0, 0, 100, 98, -98, 13, -12, 42]
    return np.array(vals, np.float32), np.array(codes, np.int8)


def test_q8_1_hand_block_closed_form(oracle_mod):
    x, codes = _q8_1_hand_block()
    q, d, s = oracle_mod.quantize_q8_1(x, 32, 1)
    assert d[0, 0] == np.float32(1.0)
    assert np.array_equal(q[0], codes)
    assert s[0, 0] == int(codes.astype(np.int64).sum())


@pytest.mark.parametrize("scale", [2.0 ** -10, 3.0, 2.0 ** 40, 2.0 ** -100])
def test_q8_1_exact_multiples(oracle_mod, scale):
    """x = c*k with integer codes k and max |k| = 127: d = c and q = k exactly."""
    rng = np.random.default_rng(7)
    k = rng.integers(-127, 128, size=(3, 64)).astype(np.int64)
    k[:, 0] = 127
    k[:, 32] = -127
    x = (k * scale).astype(np.float32)
    assert np.array_equal(x.astype(np.float64), k * scale)      # representable
    q, d, s = oracle_mod.quantize_q8_1(x, 64, 3)
    assert np.array_equal(d, np.full((3, 2), scale, np.float32))
    assert np.array_equal(q.astype(np.int64), k)
    assert np.array_equal(s, k.reshape(3, 2, 32).sum(-1))


def test_q8_1_zero_and_non_finite_blocks(oracle_mod):
    x = qsynth.make_x(1, 160, seed=3).copy()
    x[0, 0:32] = 0.0
    x[0, 40] = np.nan
    x[0, 70] = -np.inf
    x[0, 100] = np.inf
    q, d, s = oracle_mod.quantize_q8_1(x, 160, 1)
    assert d[0, 0] == 0.0 and not q[0, :32].any() and s[0, 0] == 0
    for j in (1, 2, 3):
        assert np.isnan(d[0, j]) and not q[0, 32 * j:32 * j + 32].any() and s[0, j] == 0
    assert np.isfinite(d[0, 4]) and d[0, 4] > 0


def test_q8_1_subnormal_scale_clamps(oracle_mod):
    """amax = 190 * 2^-149 (subnormal): d = 190/127 ulp rounds to one ulp,
    2^-149, so x/d reaches 190 for the largest entry and must clamp to 127;
    the small entries are exact multiples of d and keep their codes."""
    u = np.float32(2.0 ** -149)
    k = np.arange(-16, 16, dtype=np.int64)
    x = (k * np.float64(u)).astype(np.float32)
    x[0] = np.float32(190) * u
    x[1] = -np.float32(190) * u
    q, d, s = oracle_mod.quantize_q8_1(x, 32, 1)
    assert d[0, 0] == u
    expect = k.copy()
    expect[0], expect[1] = 127, -127
    assert np.array_equal(q[0].astype(np.int64), expect)
    assert s[0, 0] == expect.sum()


def test_q8_1_against_numpy_rounding(oracle_mod):
    """Random blocks over many magnitudes: d is the fp32 quotient amax/127,
    codes are numpy's round-half-even of the fp32 quotient x/d (an independent
    rounding routine), the reconstruction error is at most d/2 (plus the
    quotient's own rounding), every block reaches |q| = 127 and the codes are
    odd in x."""
    rng = np.random.default_rng(11)
    batch, ncols = 4, 2048
    x = (rng.standard_normal((batch, ncols)) *
         np.exp2(rng.integers(-60, 60, size=(batch, ncols // 32, 1)).repeat(32, -1).reshape(batch, ncols))
         ).astype(np.float32)
    q, d, s = oracle_mod.quantize_q8_1(x, ncols, batch)
    xb = x.reshape(batch, -1, 32)
    amax = np.abs(xb).max(-1)
    assert np.array_equal(d, (amax / np.float32(127)).astype(np.float32))
    with np.errstate(invalid="ignore", divide="ignore"):
        t = (xb / d[..., None]).astype(np.float32)
    ref = np.clip(np.rint(t), -127, 127).astype(np.int8)
    assert np.array_equal(q.reshape(batch, -1, 32), ref)
    assert np.array_equal(s, q.reshape(batch, -1, 32).astype(np.int64).sum(-1))
    err = np.abs(xb.astype(np.float64) - d[..., None].astype(np.float64) * q.reshape(batch, -1, 32))
    assert np.all(err <= d[..., None].astype(np.float64) * (0.5 + 2.0 ** -16))
    assert np.all(np.abs(q.reshape(batch, -1, 32)).max(-1) == 127)
    qn, dn, sn = oracle_mod.quantize_q8_1(-x, ncols, batch)
    assert np.array_equal(qn, -q) and np.array_equal(dn, d) and np.array_equal(sn, -s)


@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q8_0"])
def test_gemv_q8_1_equals_gemv_on_representable_x(oracle_mod, fmt):
    """When every x is a code times its block's scale, quantizing loses
    nothing, so the quantized-activation GEMV equals the plain GEMV bit for bit
    (the plain GEMV is pinned above).  Scales differ per block, which pins the
    block index of d."""
    nrows, ncols, batch = 7, 256, 3
    rng = np.random.default_rng(13)
    k = rng.integers(-127, 128, size=(batch, ncols // 32, 32)).astype(np.int64)
    k[:, :, 5] = 127
    c = np.exp2(rng.integers(-8, 8, size=(batch, ncols // 32, 1))).astype(np.float64)
    x = (k * c).reshape(batch, ncols).astype(np.float32)
    W = qsynth.make_weights(fmt, nrows, ncols, seed=17)
    q, d, _ = oracle_mod.quantize_q8_1(x, ncols, batch)
    assert np.array_equal(d, c[..., 0].astype(np.float32))
    yq, abq = oracle_mod.gemv_q8_1(fmt, W, q, d, nrows, ncols, batch)
    y, ab = oracle_mod.gemv(fmt, W, x, nrows, ncols, batch)
    assert np.array_equal(yq, y) and np.array_equal(abq, ab)


def _raw_blocks(fmt, W, nrows, ncols):
    """Numpy decode of the raw block fields (scale fields and integer codes)."""
    bb = {"q4_0": 18, "q4_1": 20, "q8_0": 34}[fmt]
    raw = np.asarray(W, np.uint8).reshape(nrows, ncols // 32, bb)
    d = raw[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    if fmt == "q8_0":
        return d, None, raw[..., 2:].view(np.int8).astype(np.int64)
    qs = raw[..., 4:] if fmt == "q4_1" else raw[..., 2:]
    codes = np.concatenate([qs & 15, qs >> 4], -1).astype(np.int64)
    if fmt == "q4_0":
        return d, None, codes - 8
    m = raw[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    return d, m, codes


@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q8_0"])
def test_gemv_q8_1_integer_form(oracle_mod, fmt):
    """The integer-dot form a byte-wise dot product kernel evaluates:
    y = sum_j dx_j * (d_j * sum_i qw_i qx_i  [+ m_j * sum_i qx_i for Q4_1]),
    computed here with int64 codes from a numpy decode of the raw bytes."""
    nrows, ncols, batch = 9, 512, 2
    W = qsynth.make_weights(fmt, nrows, ncols, seed=19)
    x = qsynth.make_x(batch, ncols, seed=20)
    q, d, s = oracle_mod.quantize_q8_1(x, ncols, batch)
    yq, abq = oracle_mod.gemv_q8_1(fmt, W, q, d, nrows, ncols, batch)
    dw, mw, cw = _raw_blocks(fmt, W, nrows, ncols)
    qx = q.reshape(batch, 1, ncols // 32, 32).astype(np.int64)
    sumi = (cw[None] * qx).sum(-1)                                   # [batch][nrows][nb]
    terms = dw[None] * sumi
    if mw is not None:
        terms = terms + mw[None] * s[:, None, :]
    ref = (terms * d[:, None, :].astype(np.float64)).sum(-1)
    tol = 2.0 ** -22 * abq + 1e-30
    assert np.all(np.abs(yq.astype(np.float64) - ref) <= tol)


def test_gemv_q8_1_one_hot_and_nan(oracle_mod):
    nrows, ncols = 5, 96
    W = qsynth.make_weights("q8_0", nrows, ncols, seed=23)
    w = oracle_mod.dequant("q8_0", W, nrows, ncols).astype(np.float64)
    q = np.zeros((2, ncols), np.int8)
    d = np.ones((2, 3), np.float32)
    q[0, 37] = 127
    d[1, 2] = np.nan
    y, _ = oracle_mod.gemv_q8_1("q8_0", W, q, d, nrows, ncols, 2)
    assert np.array_equal(y[0].astype(np.float64), 127.0 * w[:, 37])
    assert np.all(np.isnan(y[1]))


@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q8_0"])
def test_gemv_q8_1_error_bound(oracle_mod, fmt):
    """The quantized-activation GEMV stays within its stated distance of the
    plain GEMV: |y_q - y| <= sum_j (amax_j / 254) * sum_{i in j} |w_i| * (1 + 2^-14)
    + 2^-22 * (sum|w x| + sum|w xhat|), per output."""
    nrows, ncols, batch = 11, 1024, 3
    W = qsynth.make_weights(fmt, nrows, ncols, seed=29)
    x = qsynth.make_x(batch, ncols, seed=30).copy()
    x[1] *= np.exp2(np.arange(ncols) % 40 - 20).astype(np.float32)      # mixed magnitudes
    q, d, _ = oracle_mod.quantize_q8_1(x, ncols, batch)
    yq, abq = oracle_mod.gemv_q8_1(fmt, W, q, d, nrows, ncols, batch)
    y, ab = oracle_mod.gemv(fmt, W, x, nrows, ncols, batch)
    aw = np.abs(oracle_mod.dequant(fmt, W, nrows, ncols).astype(np.float64)).reshape(nrows, -1, 32).sum(-1)
    amax = np.abs(x.astype(np.float64)).reshape(batch, -1, 32).max(-1)
    bound = (amax[:, None, :] / 254.0 * aw[None]).sum(-1) * (1 + 2.0 ** -14) + 2.0 ** -22 * (ab + abq)
    err = np.abs(yq.astype(np.float64) - y.astype(np.float64))
    assert np.all(err <= bound)
    assert err.max() > 0                                                 # the bound is not vacuous



# --------------------------------------------------------- expert-selected GEMV

def test_gemv_id_selects_expert_matrices(oracle_mod):
    """Each batch column equals the plain GEMV of its own expert's matrix
    (cut from the stack by byte offset in the test), including repeated and
    unused experts; an id out of range is rejected."""
    nrows, ncols, ne = 7, 192, 5
    for fmt in ("q4_0", "q4_1", "q8_0"):
        W = qsynth.make_weights(fmt, nrows * ne, ncols, seed=91)
        ebytes = nrows * (ncols // 32) * {"q4_0": 18, "q4_1": 20, "q8_0": 34}[fmt]
        ids = np.array([3, 0, 3, 4], np.int32)
        x = qsynth.make_x(4, ncols, seed=92)
        y, ab = oracle_mod.gemv_id(fmt, W, ne, ids, x, nrows, ncols, 4)
        for b, e in enumerate(ids):
            ye, abe = oracle_mod.gemv(fmt, W[e * ebytes:(e + 1) * ebytes], x[b:b + 1], nrows, ncols, 1)
            assert np.array_equal(y[b], ye[0]) and np.array_equal(ab[b], abe[0])
        # brute force on the decoded stack
        w = oracle_mod.dequant(fmt, W, nrows * ne, ncols).astype(np.float64).reshape(ne, nrows, ncols)
        ref = np.einsum("brk,bk->br", w[ids], x.astype(np.float64))
        assert np.allclose(y, ref.astype(np.float32), rtol=1e-6, atol=1e-12)
        with pytest.raises(ValueError):
            oracle_mod.gemv_id(fmt, W, ne, np.array([0, 5, 0, 0], np.int32), x, nrows, ncols, 4)
        with pytest.raises(ValueError):
            oracle_mod.gemv_id(fmt, W, ne, np.array([0, -1, 0, 0], np.int32), x, nrows, ncols, 4)
        # shared activations: columns 2t and 2t+1 read row t, as if each of
        # them had its own copy of it
        x2 = qsynth.make_x(2, ncols, seed=93)
        yg, abg = oracle_mod.gemv_id(fmt, W, ne, ids, x2, nrows, ncols, 4, x_group=2)
        yr, abr = oracle_mod.gemv_id(fmt, W, ne, ids, np.repeat(x2, 2, axis=0), nrows, ncols, 4)
        assert np.array_equal(yg, yr) and np.array_equal(abg, abr)
        assert not np.array_equal(yg[1], yg[2])
        with pytest.raises(ValueError):
            oracle_mod.gemv_id(fmt, W, ne, ids[:3], x2, nrows, ncols, 3, x_group=2)
