"""GPU parity of the standalone dequantization against the CPU oracle:
bit-exact fp32 and fp16 outputs, through the C ABI.

Shapes: the small correctness matrix (64 x 256, 8 blocks per row), ragged
sizes whose block count is not a multiple of the kernel's 32-block group, and
the full 4096 x 32768 (2^27-element) tensor in Q4_0 and Q8_0 that the
benchmark times.  Special scales (+-0, subnormal, largest fp16, infinity) and
Q8_0 code -128 are covered too."""
import numpy as np
import pytest

import qsynth
from gpu_util import bf16_dev, qlib, to_dev, torch_cuda, weights

pytestmark = pytest.mark.gpu

FMTS = ["q4_0", "q4_1", "q8_0"]


def run_dequant(q, torch, fmt, Wn, nrows, ncols, f16):
    W = to_dev(Wn, torch)
    out = torch.full((nrows, ncols), float("nan"), dtype=torch.float16 if f16 else torch.float32, device="cuda")
    getattr(q, "qdequant_" + fmt)(W, out, nrows, ncols)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    return out.cpu().numpy()


def check_bits(got, ref, f16):
    g = got.view(np.uint16 if f16 else np.uint32)
    r = ref.view(np.uint16) if f16 else ref.view(np.uint32)
    if f16:
        gn = np.isnan(got.astype(np.float32))
        rn = np.isnan(ref.view(np.float16).astype(np.float32))
    else:
        gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn)
    bad = np.nonzero((g != r) & ~gn)
    assert bad[0].size == 0, "first mismatches at %s" % (list(zip(*[b[:5] for b in bad])),)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("shape", [(64, 256), (1, 32), (3, 96), (7, 1056), (33, 544), (130, 4096)])
def test_dequant_bit_exact(oracle_mod, fmt, f16, shape):
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = shape
    Wn = weights(fmt, nrows, ncols, 1000 + nrows)
    got = run_dequant(q, torch, fmt, Wn, nrows, ncols, f16)
    ref = oracle_mod.dequant(fmt, Wn, nrows, ncols, out="f16" if f16 else "f32")
    check_bits(got, ref, f16)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("f16", [False, True])
def test_dequant_full_2p27(oracle_mod, fmt, f16):
    """The 2^27-element tensor (4096 x 32768), every element compared."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = 4096, 32768
    Wn = weights(fmt, nrows, ncols, 3000)
    got = run_dequant(q, torch, fmt, Wn, nrows, ncols, f16)
    ref = oracle_mod.dequant(fmt, Wn, nrows, ncols, out="f16" if f16 else "f32")
    check_bits(got, ref, f16)


def special_blocks(fmt):
    scales = np.array([0.0, -0.0, 2.0**-24, 6.1e-5, 65504.0, -65504.0, 1.0, np.inf], np.float16)
    g = qsynth.rng(77)
    n = scales.size * 4
    d = np.repeat(scales, 4)
    if fmt == "q8_0":
        qs = g.integers(-128, 128, (n, 32)).astype(np.int8)
        qs[:, 0] = -128
        qs[:, 1] = 127
        return qsynth.pack_blocks(fmt, d, qs), n
    qs = g.integers(0, 256, (n, 16), dtype=np.uint8)
    qs[:, 0] = 0x00
    qs[:, 1] = 0xFF
    qs[:, 2] = 0x88
    m = None
    if fmt == "q4_1":
        m = np.tile(np.array([0.0, -0.0, -0.08, 2.0**-20], np.float16), scales.size)
    return qsynth.pack_blocks(fmt, d, qs, m), n


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("f16", [False, True])
def test_dequant_special_scales(oracle_mod, fmt, f16):
    torch = torch_cuda()
    q = qlib()
    Wn, n = special_blocks(fmt)
    got = run_dequant(q, torch, fmt, Wn, n, 32, f16)
    ref = oracle_mod.dequant(fmt, Wn, n, 32, out="f16" if f16 else "f32")
    check_bits(got, ref, f16)


def test_dequant_writes_nothing_outside(oracle_mod):
    """Guard bands around the output stay untouched (ragged block count)."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = 5, 288                     # 45 blocks: one full group + a 13-block tail
    Wn = weights("q4_0", nrows, ncols, 4242)
    W = to_dev(Wn, torch)
    guard = 1024
    buf = torch.full((guard + nrows * ncols + guard,), -7.0, dtype=torch.float32, device="cuda")
    out = buf[guard:guard + nrows * ncols]
    q.qdequant_q4_0(W, out, nrows, ncols)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:guard] == -7.0) and np.all(b[guard + nrows * ncols:] == -7.0)
    ref = oracle_mod.dequant("q4_0", Wn, nrows, ncols)
    assert np.array_equal(b[guard:guard + nrows * ncols].view(np.uint32), ref.reshape(-1).view(np.uint32))


def test_dequant_rejects_misaligned_output():
    torch = torch_cuda()
    q = qlib()
    W = to_dev(weights("q4_0", 2, 64, 1), torch)
    buf = torch.zeros(2 * 64 + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QgemvError) as e:
        q.qdequant_q4_0(W, buf[1:1 + 128], 2, 64)
    assert e.value.status == 4
