"""GPU parity of the GEMV against the CPU oracle, through the C ABI.

Bar: |y_gpu - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-6 for every element.
Shapes: the 64 x 256 correctness case, the 4096 x 4096 attention projection,
both FFN shapes (14336 x 4096 and 4096 x 14336) in all three formats at batch
1, 2, 4 and 8 (every element compared), plus edge shapes: a single block,
ragged row counts, ncols not a multiple of 256, odd batches, empty inputs.
Also checks determinism (bitwise equal repeated calls) and guard bands."""
import numpy as np
import pytest

import qsynth
from gpu_util import assert_within_bound, qlib, to_dev, torch_cuda, weights

pytestmark = pytest.mark.gpu

FMTS = ["q4_0", "q4_1", "q8_0"]


def run_gemv(q, torch, fmt, Wn, xn, nrows, ncols, batch, W=None):
    if W is None:
        W = to_dev(Wn, torch)
    x = to_dev(xn, torch)
    y = torch.full((batch, nrows), float("nan"), dtype=torch.float32, device="cuda")
    getattr(q, "qgemv_" + fmt)(W, x, y, nrows, ncols, batch)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    return y.cpu().numpy()


def check(oracle_mod, q, torch, fmt, nrows, ncols, batch, seed):
    Wn = weights(fmt, nrows, ncols, seed)
    xn = qsynth.make_x(batch, ncols, seed + 1)
    got = run_gemv(q, torch, fmt, Wn, xn, nrows, ncols, batch)
    ref, ab = oracle_mod.gemv(fmt, Wn, xn, nrows, ncols, batch)
    return assert_within_bound(got, ref, ab, "%s %dx%d b%d" % (fmt, nrows, ncols, batch))


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_small_config(oracle_mod, fmt):
    torch = torch_cuda()
    check(oracle_mod, qlib(), torch, fmt, 64, 256, 1, 0)


def test_gemv_attention_projection(oracle_mod):
    torch = torch_cuda()
    check(oracle_mod, qlib(), torch, "q4_0", 4096, 4096, 1, 10)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(14336, 4096), (4096, 14336)])
@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_gemv_ffn_shapes(oracle_mod, fmt, shape, batch):
    torch = torch_cuda()
    nrows, ncols = shape
    check(oracle_mod, qlib(), torch, fmt, nrows, ncols, batch, 20)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape,batch", [((1, 32), 1), ((3, 96), 2), ((17, 800), 3), ((5, 256), 8),
                                         ((129, 512), 5), ((31, 1056), 7), ((1000, 288), 6),
                                         ((2, 14336), 1), ((300, 4128), 4)])
def test_gemv_edge_shapes(oracle_mod, fmt, shape, batch):
    torch = torch_cuda()
    check(oracle_mod, qlib(), torch, fmt, shape[0], shape[1], batch, 30 + shape[0])


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_deterministic(fmt):
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, batch = 4096, 14336, 2
    Wn = weights(fmt, nrows, ncols, 20)
    xn = qsynth.make_x(batch, ncols, 99)
    W = to_dev(Wn, torch)
    a = run_gemv(q, torch, fmt, Wn, xn, nrows, ncols, batch, W=W)
    b = run_gemv(q, torch, fmt, Wn, xn, nrows, ncols, batch, W=W)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_gemv_special_inputs(oracle_mod):
    """Zero scales, subnormal scales, one-hot and all-zero activations."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = 40, 512
    g = qsynth.rng(5)
    nblk = nrows * ncols // 32
    d = g.uniform(1e-3, 1e-2, nblk).astype(np.float16)
    d[::7] = 0.0
    d[3::11] = np.float16(2.0**-24)
    qs = g.integers(0, 256, (nblk, 16), dtype=np.uint8)
    Wn = qsynth.pack_blocks("q4_0", d, qs)
    xn = np.zeros((4, ncols), np.float32)
    xn[0, 17] = 1.0
    xn[2] = qsynth.make_x(1, ncols, 6)[0]
    xn[3, :] = 1e30                      # large activations stay finite in fp32 accumulation
    got = run_gemv(q, torch, "q4_0", Wn, xn, nrows, ncols, 4)
    ref, ab = oracle_mod.gemv("q4_0", Wn, xn, nrows, ncols, 4)
    assert_within_bound(got, ref, ab, "special")
    assert np.array_equal(got[1], np.zeros(nrows, np.float32))


def test_gemv_writes_only_y():
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, batch = 77, 256, 3
    W = to_dev(weights("q8_0", nrows, ncols, 8), torch)
    x = to_dev(qsynth.make_x(batch, ncols, 9), torch)
    guard = 256
    buf = torch.full((2 * guard + batch * nrows,), -3.0, dtype=torch.float32, device="cuda")
    q.qgemv_q8_0(W, x, buf[guard:guard + batch * nrows], nrows, ncols, batch)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:guard] == -3.0) and np.all(b[guard + batch * nrows:] == -3.0)


def test_gemv_empty_and_errors():
    torch = torch_cuda()
    q = qlib()
    W = to_dev(weights("q4_0", 4, 64, 1), torch)
    x = torch.zeros(1, 64, device="cuda")
    y = torch.full((1, 4), 5.0, device="cuda")
    q.qgemv_q4_0(W, x, y, 0, 64, 1)                 # empty: nothing written
    torch.cuda.synchronize()
    assert torch.all(y == 5.0)
    xb = torch.zeros(9, 64, device="cuda")
    yb = torch.zeros(9, 4, device="cuda")
    with pytest.raises(q.QgemvError) as e:
        q.qgemv_q4_0(W, xb, yb, 4, 64, 9)
    assert e.value.status == 3
    with pytest.raises(q.QgemvError) as e:
        q.qgemv_q4_0(W, x, y, 4, 48, 1)
    assert e.value.status == 2
