"""GPU parity of the quantized-activation GEMV family (mul_mat_vec_q: the
ggml_cuda_op_mul_mat_vec_q hunk and the convert_src1_to_q8_1 flag of
ggml_cuda_op_mul_mat on the "llama_cpp 0.12.1 -> 0.12.2" page), through the
C ABI, against the oracle's quantize_q8_1 / gemv_q8_1.

* qquantize_q8_1 is compared bit for bit: codes, scales (NaN where the
  oracle's is NaN) and code sums.  Decisions (the codes) are taken in fp32 on
  both sides, by IEEE division and round-half-even.
* qgemv_mmvq_* is compared element by element with the oracle's GEMV over
  the oracle's own quantized activations at |y - y_ref| <= 1e-5 * sum_k
  |w_k xhat_k| + 1e-30 (fp32 accumulation of exact integer block sums), and
  with the plain GEMV of x at the bound the activation rounding allows.
* Special weights and activations, guard bands, determinism and the
  timeout path, as for the fp32-activation GEMV.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import qsynth
from gpu_util import qlib, to_dev, torch_cuda
from test_gpu_special import run_guarded, special_weights, special_x

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
FMTS = ["q4_0", "q4_1", "q8_0"]
TOL_REL = 1e-5
TOL_ABS = 1e-30


def assert_mmvq_close(got, ref, absdot, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "%s: NaN positions differ" % what
    err = np.abs(got[~nan] - ref[~nan])
    bound = TOL_REL * np.asarray(absdot)[~nan] + TOL_ABS
    bad = ~(err <= bound)
    assert not bad.any(), "%s: %d elements outside the bound; got %s ref %s bound %s" % (
        what, int(bad.sum()), got[~nan][bad][:5], ref[~nan][bad][:5], bound[bad][:5])
    return float((err / bound).max()) if err.size else 0.0


def pack_xq(q, d, s):
    """The quantized-activation buffer layout: codes, then scales, then sums."""
    return np.concatenate([np.ascontiguousarray(q).view(np.uint8).ravel(),
                           np.ascontiguousarray(d, np.float32).view(np.uint8).ravel(),
                           np.ascontiguousarray(s, np.int32).view(np.uint8).ravel()])


def q8_special_x(batch, ncols, seed):
    """Blocks over many binades, zero / NaN / infinite blocks, round-half ties
    (a block whose amax is 127, so that d = 1 and x/d = x), and a block whose
    subnormal amax makes the code 190 before the clamp."""
    g = np.random.default_rng(seed)
    nb = ncols // 32
    x = g.standard_normal((batch, nb, 32)).astype(np.float32)
    x *= np.exp2(g.integers(-100, 100, size=(batch, nb, 1))).astype(np.float32)
    ties = np.array([127.0, -127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, -3.5, 126.5, -126.5,
                     0.0, -0.0, 100.5, -100.5, 5.5, 6.5, -5.5, -6.5, 64.5, -64.5, 7.5, 8.5,
                     99.5, 98.5, -98.5, 12.5, -12.5, 42.5, 0.49999997, 1e-30], np.float32)
    u = np.float32(2.0 ** -149)
    sub = (np.arange(-16, 16) * np.float64(u)).astype(np.float32)
    sub[0], sub[1] = 190 * u, -190 * u
    for b in range(batch):
        sel = [j for j in range(nb)]
        if nb > 1:
            x[b, sel[1]] = 0.0
        if nb > 2:
            x[b, sel[2]] = ties
        if nb > 3:
            x[b, sel[3]] = sub
        if nb > 4 and b % 2 == 0:
            x[b, sel[4], 9] = np.nan
        if nb > 5 and b % 3 == 0:
            x[b, sel[5], 30] = -np.inf
    return x.reshape(batch, ncols)


def gpu_quantize(q, torch, xn, ncols, batch):
    xq = torch.empty(q.q8_1_size(ncols, batch), dtype=torch.uint8, device="cuda")
    q.qquantize_q8_1(to_dev(xn, torch), xq, ncols, batch)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    return xq


@pytest.mark.parametrize("batch,ncols", [(1, 64), (3, 256), (8, 4096), (1, 14336), (2, 14336), (5, 96)])
@pytest.mark.parametrize("kind", ["normal", "special"])
def test_quantize_bit_exact(oracle_mod, batch, ncols, kind):
    torch = torch_cuda()
    q = qlib()
    if kind == "normal":
        xn = qsynth.make_x(batch, ncols, seed=batch * 31 + ncols)
    else:
        xn = q8_special_x(batch, ncols, seed=batch + ncols)
    xq = gpu_quantize(q, torch, xn, ncols, batch)
    codes, d, s = q.q8_1_views(xq, ncols, batch)
    rq, rd, rs = oracle_mod.quantize_q8_1(xn, ncols, batch)
    assert np.array_equal(codes.cpu().numpy(), rq)
    dg = d.cpu().numpy()
    assert np.array_equal(np.isnan(dg), np.isnan(rd))
    ok = ~np.isnan(rd)
    assert np.array_equal(dg[ok].view(np.uint32), rd[ok].view(np.uint32))
    assert np.array_equal(s.cpu().numpy(), rs)


CASES = [(64, 256, 1), (77, 2048, 1), (77, 2048, 3), (300, 1024, 8), (1000, 4096, 2), (5, 96, 2),
         (33, 128, 4), (130, 640, 7), (4096, 14336, 1), (14336, 4096, 8)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("nrows,ncols,batch", CASES)
def test_mmvq_matches_oracle(oracle_mod, fmt, nrows, ncols, batch):
    torch = torch_cuda()
    q = qlib()
    Wn = qsynth.make_weights(fmt, nrows, ncols, seed=nrows + 3 * ncols)
    xn = qsynth.make_x(batch, ncols, seed=batch + 7)
    W, x = to_dev(Wn, torch), to_dev(xn, torch)
    rq, rd, rs = oracle_mod.quantize_q8_1(xn, ncols, batch)
    ref, ab = oracle_mod.gemv_q8_1(fmt, Wn, rq, rd, nrows, ncols, batch)
    # the one-call form (quantizes inside the call)
    y = torch.full((batch, nrows), float("nan"), device="cuda")
    getattr(q, "qgemv_mmvq_" + fmt)(W, x, y, nrows, ncols, batch)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    got = y.cpu().numpy()
    assert_mmvq_close(got, ref, ab, "%s %dx%d b%d" % (fmt, nrows, ncols, batch))
    # the GEMV alone on the oracle's quantized activations gives the same bits
    xq = to_dev(pack_xq(rq, rd, rs), torch)
    y2 = torch.full((batch, nrows), float("nan"), device="cuda")
    getattr(q, "qgemv_mmvq_xq_" + fmt)(W, xq, y2, nrows, ncols, batch)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), got.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("nrows,ncols,batch", [(77, 2048, 1), (77, 2048, 7), (300, 4096, 3), (4096, 14336, 8),
                                               (21, 96, 5)])
def test_mmvq_special_values(oracle_mod, fmt, nrows, ncols, batch):
    """Scales d = +0, -0 and 2^-24, Q8_0 codes -128, zero rows, activations
    zero / one-hot / 1e11 spikes / 1e-30 and 1e30 scaled, guard bands."""
    torch = torch_cuda()
    q = qlib()
    kstar = ncols // 2 + 37
    Wn, blank = special_weights(fmt, nrows, ncols, 50 + nrows, kstar)
    xn, kinds = special_x(batch, ncols, 51, kstar)
    if batch == 1:
        xn[0, kstar] = 1e11
    W, x = to_dev(Wn, torch), to_dev(xn, torch)
    got = run_guarded(q, torch, getattr(q, "qgemv_mmvq_" + fmt),
                      lambda out: (W, x, out.view(batch, nrows), nrows, ncols, batch), batch * nrows)
    got = got.reshape(batch, nrows)
    rq, rd, _ = oracle_mod.quantize_q8_1(xn, ncols, batch)
    ref, ab = oracle_mod.gemv_q8_1(fmt, Wn, rq, rd, nrows, ncols, batch)
    assert_mmvq_close(got, ref, ab, "%s %dx%d b%d special" % (fmt, nrows, ncols, batch))
    assert np.all(got[:, blank] == 0.0)
    for n, kind in enumerate(kinds):
        if kind == 1:
            assert np.all(got[n] == 0.0)


@pytest.mark.parametrize("fmt", FMTS)
def test_mmvq_non_finite_activations(oracle_mod, fmt):
    """A block of x holding a NaN or an infinity has d = NaN: every row of that
    batch column is NaN; the other columns are unaffected."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, batch = 300, 4096, 3
    Wn = qsynth.make_weights(fmt, nrows, ncols, seed=61)
    xn = qsynth.make_x(batch, ncols, seed=62).copy()
    xn[0, 1000] = np.nan
    xn[2, 5] = np.inf
    y = torch.empty(batch, nrows, device="cuda")
    getattr(q, "qgemv_mmvq_" + fmt)(to_dev(Wn, torch), to_dev(xn, torch), y, nrows, ncols, batch)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    assert np.all(np.isnan(got[0])) and np.all(np.isnan(got[2])) and np.all(np.isfinite(got[1]))
    rq, rd, _ = oracle_mod.quantize_q8_1(xn, ncols, batch)
    ref, ab = oracle_mod.gemv_q8_1(fmt, Wn, rq, rd, nrows, ncols, batch)
    assert_mmvq_close(got, ref, ab, "non-finite x")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("nrows,ncols,batch", [(4096, 14336, 1), (14336, 4096, 4)])
def test_mmvq_error_against_plain_gemv(oracle_mod, fmt, nrows, ncols, batch):
    """The quantized-activation result stays within the activation-rounding
    bound of the plain GEMV of x:
    |y - y_plain| <= sum_j (amax_j / 254) * sum_{k in j} |w_k| * (1 + 2^-14)
                     + 1e-5 * sum_k |w_k xhat_k| + 2^-20 * sum_k |w_k x_k| + 1e-30."""
    torch = torch_cuda()
    q = qlib()
    Wn = qsynth.make_weights(fmt, nrows, ncols, seed=71 + nrows)
    xn = qsynth.make_x(batch, ncols, seed=72)
    y = torch.empty(batch, nrows, device="cuda")
    getattr(q, "qgemv_mmvq_" + fmt)(to_dev(Wn, torch), to_dev(xn, torch), y, nrows, ncols, batch)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    plain, ab = oracle_mod.gemv(fmt, Wn, xn, nrows, ncols, batch)
    rq, rd, _ = oracle_mod.quantize_q8_1(xn, ncols, batch)
    _, abq = oracle_mod.gemv_q8_1(fmt, Wn, rq, rd, nrows, ncols, batch)
    aw = np.abs(oracle_mod.dequant(fmt, Wn, nrows, ncols).astype(np.float64)).reshape(nrows, -1, 32).sum(-1)
    amax = np.abs(xn.astype(np.float64)).reshape(batch, -1, 32).max(-1)
    bound = ((amax[:, None, :] / 254.0) * aw[None]).sum(-1) * (1 + 2.0 ** -14) + TOL_REL * abq \
        + 2.0 ** -20 * ab + TOL_ABS
    err = np.abs(got - plain)
    assert np.all(err <= bound)
    rel = err / ab
    print("%s %dx%d b%d: activation rounding error / sum|w x|: max %.3g median %.3g; / bound max %.3g" % (
        fmt, nrows, ncols, batch, rel.max(), np.median(rel), (err / bound).max()))


@pytest.mark.parametrize("fmt", FMTS)
def test_mmvq_deterministic(fmt):
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, batch = 4096, 14336, 3
    Wn = qsynth.make_weights(fmt, nrows, ncols, seed=5)
    xn = q8_special_x(batch, ncols, seed=6)
    W, x = to_dev(Wn, torch), to_dev(xn, torch)
    outs = []
    for _ in range(3):
        y = torch.empty(batch, nrows, device="cuda")
        getattr(q, "qgemv_mmvq_" + fmt)(W, x, y, nrows, ncols, batch)
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy().view(np.uint32))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_mmvq_wait_timeout_reported_and_recovered(oracle_mod):
    """The streaming kernel's first weight copy withheld: its waits give up,
    qgemv_sync_check reports QGEMV_ERR_TIMEOUT, and the next call is correct."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols = 512, 4096
    Wn = qsynth.make_weights("q4_0", nrows, ncols, 87)
    xn = qsynth.make_x(1, ncols, 88)
    W, x = to_dev(Wn, torch), to_dev(xn, torch)
    y = torch.empty(1, nrows, device="cuda")
    q.qgemv_set_option(q.OPT_WAIT_PROBES, 2000)
    try:
        q.qgemv_set_option(q.OPT_TEST_WITHHOLD_COPY, 1)
        q.qgemv_mmvq_q4_0(W, x, y, nrows, ncols, 1)
        with pytest.raises(q.QgemvError) as e:
            q.qgemv_sync_check()
        assert e.value.status == 8
    finally:
        q.qgemv_set_option(q.OPT_WAIT_PROBES, 1 << 20)
        q.qgemv_set_option(q.OPT_TEST_WITHHOLD_COPY, 0)
    rq, rd, _ = oracle_mod.quantize_q8_1(xn, ncols, 1)
    ref, ab = oracle_mod.gemv_q8_1("q4_0", Wn, rq, rd, nrows, ncols, 1)
    for _ in range(2):
        y.fill_(float("nan"))
        q.qgemv_mmvq_q4_0(W, x, y, nrows, ncols, 1)
        torch.cuda.synchronize()
        q.qgemv_sync_check()
        assert_mmvq_close(y.cpu().numpy(), ref, ab, "after timeout")


@pytest.mark.parametrize("path", ["stream", "rowwarp"])
def test_forced_mmvq_path_matches_oracle(path):
    """Each kernel of the family on every shape it takes, in a child process
    with QGEMV_MMVQ_PATH forcing it (read once per process)."""
    torch_cuda()
    env = dict(os.environ, QGEMV_MMVQ_PATH=path)
    r = subprocess.run([sys.executable, os.path.join(HERE, "mmvq_path_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
