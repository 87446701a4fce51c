"""Packed Q4_0 GEMV path (qgemv_pack_q4_0 + qgemv_packed_q4_0) through the C
ABI: the packed bytes equal a numpy restatement of the layout documented in
qgemv.h (bit-exact, including the zero rows of a ragged last tile), and the
GEMV on packed weights matches the CPU oracle run on the original ggml blocks
within |y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-6 per element."""
import numpy as np
import pytest

import qsynth
from gpu_util import assert_within_bound, qlib, to_dev, torch_cuda, weights

pytestmark = pytest.mark.gpu


def pack_reference(Wn, nrows, ncols):
    """The packed order as qgemv.h states it, written with numpy indexing."""
    nb = ncols // 32
    ntiles = (nrows + 15) // 16
    npairs = nb // 2
    blocks = np.zeros((ntiles * 16, nb, 18), np.uint8)
    blocks[:nrows] = Wn.reshape(nrows, nb, 18)
    qs = blocks[:, :, 2:].reshape(ntiles, 16, npairs, 2, 16)     # [t][row in tile][p][block in pair][byte]
    d = blocks[:, :, :2].reshape(ntiles, 16, npairs, 2, 2)
    out = np.zeros((ntiles, npairs, 576), np.uint8)
    for l in range(32):
        g, c = l >> 2, l & 3
        piece = np.stack([qs[:, g, :, 0, 4 * c:4 * c + 4], qs[:, g + 8, :, 0, 4 * c:4 * c + 4],
                          qs[:, g, :, 1, 4 * c:4 * c + 4], qs[:, g + 8, :, 1, 4 * c:4 * c + 4]], axis=2)
        out[:, :, 16 * l:16 * l + 16] = piece.reshape(ntiles, npairs, 16)
    for g in range(8):
        piece = np.stack([d[:, g, :, 0], d[:, g + 8, :, 0], d[:, g, :, 1], d[:, g + 8, :, 1]], axis=2)
        out[:, :, 512 + 8 * g:512 + 8 * g + 8] = piece.reshape(ntiles, npairs, 8)
    return out.reshape(-1)


def packed_dev(q, torch, Wn, nrows, ncols):
    W = to_dev(Wn, torch)
    Wp = torch.empty(q.qgemv_packed_bytes(nrows, ncols), dtype=torch.uint8, device="cuda")
    q.qgemv_pack_q4_0(W, Wp, nrows, ncols)
    return Wp


@pytest.mark.parametrize("shape", [(1, 64), (17, 128), (40, 1024), (300, 4096), (4096, 14336)])
def test_pack_matches_documented_layout(shape):
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = shape
    Wn = weights("q4_0", nrows, ncols, 5)
    Wp = packed_dev(q, torch, Wn, nrows, ncols)
    torch.cuda.synchronize()
    assert q.qgemv_packed_bytes(nrows, ncols) == (nrows + 15) // 16 * 16 * (ncols // 32) * 18
    assert np.array_equal(Wp.cpu().numpy(), pack_reference(Wn, nrows, ncols))


@pytest.mark.parametrize("shape,batch", [((4096, 14336), 1), ((14336, 4096), 1), ((4096, 14336), 2),
                                         ((14336, 4096), 4), ((4096, 14336), 8), ((14336, 4096), 8),
                                         ((4096, 4096), 1), ((1, 64), 1), ((17, 128), 3), ((77, 2048), 5),
                                         ((300, 4096), 7), ((33, 65536), 1)])
def test_packed_gemv_matches_oracle(oracle_mod, shape, batch):
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = shape
    Wn = weights("q4_0", nrows, ncols, 20)
    xn = qsynth.make_x(batch, ncols, 21)
    Wp = packed_dev(q, torch, Wn, nrows, ncols)
    x = to_dev(xn, torch)
    y = torch.full((batch, nrows), float("nan"), dtype=torch.float32, device="cuda")
    q.qgemv_packed_q4_0(Wp, x, y, nrows, ncols, batch)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    ref, ab = oracle_mod.gemv("q4_0", Wn, xn, nrows, ncols, batch)
    assert_within_bound(y.cpu().numpy(), ref, ab, "packed q4_0 %dx%d b%d" % (nrows, ncols, batch))


def test_packed_gemv_deterministic_and_scaled_inputs(oracle_mod):
    """Same bits on repeated calls; x spanning many binades (tiny and large
    columns) stays within the bound (per-chunk power-of-two scaling)."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, batch = 512, 8192, 3
    Wn = weights("q4_0", nrows, ncols, 22)
    xn = qsynth.make_x(batch, ncols, 23)
    xn[0] *= 1e-6
    xn[1, : ncols // 2] *= 3e3
    xn[2, ::7] = 0.0
    Wp = packed_dev(q, torch, Wn, nrows, ncols)
    x = to_dev(xn, torch)
    ys = []
    for _ in range(2):
        y = torch.empty(batch, nrows, dtype=torch.float32, device="cuda")
        q.qgemv_packed_q4_0(Wp, x, y, nrows, ncols, batch)
        ys.append(y.cpu().numpy())
    assert np.array_equal(ys[0].view(np.uint32), ys[1].view(np.uint32))
    ref, ab = oracle_mod.gemv("q4_0", Wn, xn, nrows, ncols, batch)
    assert_within_bound(ys[0], ref, ab, "packed scaled x")


def test_packed_widest_rows(oracle_mod):
    """The widest rows one CTA can stage x for (71680 columns, batch 1)."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = 16, 71680
    Wn = weights("q4_0", nrows, ncols, 24)
    xn = qsynth.make_x(1, ncols, 25)
    Wp = packed_dev(q, torch, Wn, nrows, ncols)
    x = to_dev(xn, torch)
    y = torch.full((1, nrows), float("nan"), dtype=torch.float32, device="cuda")
    q.qgemv_packed_q4_0(Wp, x, y, nrows, ncols, 1)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    ref, ab = oracle_mod.gemv("q4_0", Wn, xn, nrows, ncols, 1)
    assert_within_bound(y.cpu().numpy(), ref, ab, "packed q4_0 16x71680")


def test_packed_rejects_bad_shapes():
    torch = torch_cuda()
    q = qlib()
    lib = q.lib()
    assert lib.qgemv_packed_bytes(16, 96) == -1
    rc = lib.qgemv_packed_q4_0(None, None, None, 16, 96, 1, None)
    assert rc == 2
    rc = lib.qgemv_packed_q4_0(None, None, None, 16, 128, 9, None)
    assert rc == 3
    # one batch column of x no longer fits in a CTA's shared memory: refused on the host
    Wp = torch.empty(q.qgemv_packed_bytes(16, 71744), dtype=torch.uint8, device="cuda")
    x = torch.zeros(1, 71744, dtype=torch.float32, device="cuda")
    y = torch.zeros(1, 16, dtype=torch.float32, device="cuda")
    rc = lib.qgemv_packed_q4_0(Wp.data_ptr(), x.data_ptr(), y.data_ptr(), 16, 71744, 1, None)
    assert rc == 2
