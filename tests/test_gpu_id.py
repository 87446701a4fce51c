"""GPU parity of the expert-selected GEMV (the ggml_cuda_mul_mat_id hunk and
the GGML_OP_MUL_MAT_ID cases of the "llama_cpp 0.12.1 -> 0.12.2" page; the
ffn_*_exps expert tensors of the "backend-agnostic tensor parallelism" page)
through the C ABI, against the oracle's gemv_id:

  y[b][r] = sum_k w_{ids[b]}[r][k] * x[b / x_group][k]

element by element at the GEMV bound |y - y_ref| <= 1e-3 * sum_k |w x| +
1e-6.  Cases: one token's experts sharing its activations (x_group = experts
per token, the up/gate projections) and one row per column (the down
projection) at the full Mixtral-style sizes; many tokens whose experts repeat
(columns grouped by expert on the device); all columns on one
expert (units of up to 8 columns on the tensor cores, 4 on the fixed-point
kernel); the largest batch; shapes only the general kernel takes; special
values; ids out of range; the timeout path; each kernel forced in turn.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import qsynth
from gpu_util import assert_within_bound, qlib, to_dev, torch_cuda
from test_gpu_special import run_guarded, special_weights, special_x

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
FMTS = ["q4_0", "q4_1", "q8_0"]


def expert_stack(fmt, n_expert, nrows, ncols, seed):
    return qsynth.make_weights(fmt, n_expert * nrows, ncols, seed)


def run_id(q, torch, fmt, W, n_expert, ids, x, nrows, ncols, batch, x_group):
    return run_guarded(q, torch, getattr(q, "qgemv_id_" + fmt),
                       lambda out: (W, n_expert, ids, x, out.view(batch, nrows), nrows, ncols, batch, x_group),
                       batch * nrows).reshape(batch, nrows)


def check_case(oracle_mod, fmt, nrows, ncols, n_expert, idsn, x_group, seed):
    torch = torch_cuda()
    q = qlib()
    batch = len(idsn)
    Wn = expert_stack(fmt, n_expert, nrows, ncols, seed)
    xn = qsynth.make_x(batch // x_group, ncols, seed + 1)
    idsn = np.asarray(idsn, np.int32)
    W, x, ids = to_dev(Wn, torch), to_dev(xn, torch), to_dev(idsn, torch)
    got = run_id(q, torch, fmt, W, n_expert, ids, x, nrows, ncols, batch, x_group)
    ref, ab = oracle_mod.gemv_id(fmt, Wn, n_expert, idsn, xn, nrows, ncols, batch, x_group)
    assert_within_bound(got, ref, ab, "%s %dx%d E%d b%d g%d" % (fmt, nrows, ncols, n_expert, batch, x_group))
    return got


def random_ids(n_tokens, top_k, n_expert, seed):
    """Each token's top_k distinct experts, as a router's top-k gives them."""
    g = np.random.default_rng(seed)
    return np.concatenate([g.choice(n_expert, top_k, replace=False) for _ in range(n_tokens)]).astype(np.int32)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("nrows,ncols,n_expert,ids,x_group", [
    (14336, 4096, 8, [2, 7], 2),            # one token, top-2, up/gate projection
    (4096, 14336, 8, [6, 1], 1),            # the same token's down projection
    (300, 4096, 8, [3], 1),                 # one column
    (77, 2048, 1, [0, 0, 0], 3),            # a single expert
])
def test_id_token_shapes(oracle_mod, fmt, nrows, ncols, n_expert, ids, x_group):
    check_case(oracle_mod, fmt, nrows, ncols, n_expert, ids, x_group, seed=nrows + ncols)


@pytest.mark.parametrize("fmt", FMTS)
def test_id_many_tokens_repeating_experts(oracle_mod, fmt):
    """8 tokens x top-2 of 8 experts (x_group 2) and 8 tokens x top-6 of 64
    experts (x_group 6): experts repeat across tokens and are grouped."""
    check_case(oracle_mod, fmt, 1024, 4096, 8, random_ids(8, 2, 8, 5), 2, seed=11)
    check_case(oracle_mod, fmt, 704, 2048, 64, random_ids(8, 6, 64, 6), 6, seed=12)


@pytest.mark.parametrize("fmt", FMTS)
def test_id_many_experts_token_top8(oracle_mod, fmt):
    """Many experts, one token's top-8 (DeepSeek-style FFN, hidden 7168 and
    expert width 2048): the up projection over 256 experts (2048 x 7168, 8
    columns sharing x), the down projection over 64 (7168 x 2048, one x row
    per column), then 4 tokens (32 columns) of the up projection, whose
    experts repeat."""
    check_case(oracle_mod, fmt, 2048, 7168, 256, random_ids(1, 8, 256, 71), 8, seed=72)
    ids = random_ids(1, 8, 64, 76)
    check_case(oracle_mod, fmt, 7168, 2048, 64, ids, 1, seed=73)
    check_case(oracle_mod, fmt, 2048, 7168, 64, random_ids(4, 8, 16, 74), 8, seed=75)


@pytest.mark.parametrize("fmt", FMTS)
def test_id_one_expert_units(oracle_mod, fmt):
    """Nine columns on one expert (units of 8 and 1 columns on the tensor
    cores, 4, 4 and 1 on the fixed-point kernel) all reading one activation
    row: every column is the same sum, taken in the same order whatever the
    size of its unit, so all nine come back bit for bit equal."""
    got = check_case(oracle_mod, fmt, 333, 4096, 5, [4] * 9, 9, seed=21)
    assert np.all(got == got[0])
    # and nine columns with their own rows
    check_case(oracle_mod, fmt, 333, 4096, 5, [4] * 9, 1, seed=22)


@pytest.mark.parametrize("fmt", FMTS)
def test_id_largest_batch(oracle_mod, fmt):
    g = np.random.default_rng(31)
    check_case(oracle_mod, fmt, 129, 1024, 6, g.integers(0, 6, 64).astype(np.int32), 1, seed=32)
    check_case(oracle_mod, fmt, 65, 512, 64, random_ids(8, 8, 64, 33), 8, seed=34)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("nrows,ncols", [(45, 1408), (17, 96), (9, 32), (130, 14336 + 32)])
def test_id_general_kernel_shapes(oracle_mod, fmt, nrows, ncols):
    """Row bytes not a multiple of 16 (Q4_0 / Q8_0 at 1408 or 14368 values),
    ncols not a multiple of 64, a single block: the general kernel (or the
    streaming one where the shape suits it, e.g. Q4_1 at 1408)."""
    check_case(oracle_mod, fmt, nrows, ncols, 3, [2, 0, 2, 1], 2, seed=nrows)


@pytest.mark.parametrize("fmt", FMTS)
def test_id_special_values(oracle_mod, fmt):
    """Zero, negative-zero and subnormal scales, code -128, rows of zero
    weights; activations zero, one-hot, with a 1e11 spike, with 1e-30
    values, scaled by 1e-30 and 1e30 -- one special matrix per expert."""
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, n_expert, batch = 77, 2048, 3, 7
    kstar = ncols // 2 + 37
    mats = [special_weights(fmt, nrows, ncols, 50 + e, kstar)[0] for e in range(n_expert)]
    Wn = np.concatenate(mats)
    xn, kinds = special_x(batch, ncols, 51, kstar)
    idsn = np.array([0, 2, 1, 2, 2, 0, 1], np.int32)
    W, x, ids = to_dev(Wn, torch), to_dev(xn, torch), to_dev(idsn, torch)
    got = run_id(q, torch, fmt, W, n_expert, ids, x, nrows, ncols, batch, 1)
    ref, ab = oracle_mod.gemv_id(fmt, Wn, n_expert, idsn, xn, nrows, ncols, batch, 1)
    assert_within_bound(got, ref, ab, "%s special" % fmt)
    for n, kind in enumerate(kinds):
        if kind == 1:
            assert np.all(got[n] == 0.0)


@pytest.mark.parametrize("fmt", FMTS)
def test_id_deterministic(fmt):
    torch = torch_cuda()
    q = qlib()
    nrows, ncols, n_expert = 2048, 4096, 8
    Wn = expert_stack(fmt, n_expert, nrows, ncols, 41)
    W = to_dev(Wn, torch)
    ids = to_dev(random_ids(4, 2, n_expert, 42), torch)
    x = to_dev(qsynth.make_x(4, ncols, 43), torch)
    y0 = torch.empty(8, nrows, device="cuda")
    y1 = torch.empty(8, nrows, device="cuda")
    getattr(q, "qgemv_id_" + fmt)(W, n_expert, ids, x, y0, nrows, ncols, 8, x_group=2)
    getattr(q, "qgemv_id_" + fmt)(W, n_expert, ids, x, y1, nrows, ncols, 8, x_group=2)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    assert torch.equal(y0, y1)


@pytest.mark.parametrize("ncols", [4096, 1408])
def test_id_out_of_range_ids(oracle_mod, ncols):
    """Columns with ids n_expert and -1 are left unwritten and reported as
    QGEMV_ERR_INDEX; the other columns are right; the next call is clean."""
    torch = torch_cuda()
    q = qlib()
    fmt, nrows, n_expert = "q4_0", 200, 4
    Wn = expert_stack(fmt, n_expert, nrows, ncols, 61)
    xn = qsynth.make_x(5, ncols, 62)
    idsn = np.array([1, 4, 3, -1, 1], np.int32)
    W, x, ids = to_dev(Wn, torch), to_dev(xn, torch), to_dev(idsn, torch)
    y = torch.full((5, nrows), -7.25, device="cuda")
    q.qgemv_id_q4_0(W, n_expert, ids, x, y, nrows, ncols, 5)
    with pytest.raises(q.QgemvError) as e:
        q.qgemv_sync_check()
    assert e.value.status == 11
    got = y.cpu().numpy()
    assert np.all(got[1] == -7.25) and np.all(got[3] == -7.25)
    ok = [0, 2, 4]
    ref, ab = oracle_mod.gemv_id(fmt, Wn, n_expert, idsn[ok], xn[ok], nrows, ncols, 3)
    assert_within_bound(got[ok], ref, ab, "valid columns beside bad ids")
    q.qgemv_sync_check()                          # cleared


def test_id_timeout_then_recovers(oracle_mod):
    """A withheld weight copy makes the streaming kernel's bounded wait run
    out: QGEMV_ERR_TIMEOUT, then correct results on the next calls."""
    torch = torch_cuda()
    q = qlib()
    fmt, nrows, ncols, n_expert = "q4_0", 4096, 4096, 4
    Wn = expert_stack(fmt, n_expert, nrows, ncols, 71)
    xn = qsynth.make_x(1, ncols, 72)
    idsn = np.array([3, 1], np.int32)
    W, x, ids = to_dev(Wn, torch), to_dev(xn, torch), to_dev(idsn, torch)
    y = torch.empty(2, nrows, device="cuda")
    q.qgemv_set_option(q.OPT_WAIT_PROBES, 2000)
    try:
        q.qgemv_set_option(q.OPT_TEST_WITHHOLD_COPY, 1)
        q.qgemv_id_q4_0(W, n_expert, ids, x, y, nrows, ncols, 2, x_group=2)
        with pytest.raises(q.QgemvError) as e:
            q.qgemv_sync_check()
        assert e.value.status == 8
    finally:
        q.qgemv_set_option(q.OPT_WAIT_PROBES, 1 << 20)
        q.qgemv_set_option(q.OPT_TEST_WITHHOLD_COPY, 0)
    ref, ab = oracle_mod.gemv_id(fmt, Wn, n_expert, idsn, xn, nrows, ncols, 2, 2)
    for _ in range(2):
        y.fill_(float("nan"))
        q.qgemv_id_q4_0(W, n_expert, ids, x, y, nrows, ncols, 2, x_group=2)
        torch.cuda.synchronize()
        q.qgemv_sync_check()
        assert_within_bound(y.cpu().numpy(), ref, ab, "after timeout")


def test_id_empty_problems():
    torch = torch_cuda()
    q = qlib()
    W = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    x = torch.zeros(4, 64, device="cuda")
    y = torch.full((4, 3), 5.0, device="cuda")
    q.qgemv_id_q4_0(W, 2, ids, x, y, 0, 64, 4)              # nrows == 0: nothing written
    torch.cuda.synchronize()
    assert torch.all(y == 5.0)
    q.qgemv_id_q8_0(W, 2, ids, x, y, 3, 0, 4)               # ncols == 0: zeros
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    assert torch.all(y == 0.0)


@pytest.mark.parametrize("path", ["tc", "fx", "rowwarp"])
def test_forced_id_path_matches_oracle(path):
    """Each kernel of the expert-selected GEMV (tensor cores, fixed-point
    streaming, general) on every shape it takes, in a child process with
    QGEMV_ID_PATH forcing it (read once per process)."""
    torch_cuda()
    env = dict(os.environ, QGEMV_ID_PATH=path)
    r = subprocess.run([sys.executable, os.path.join(HERE, "id_path_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
