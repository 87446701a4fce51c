"""Host-only checks of the C ABI: the library builds and loads, exports every
symbol ``include/qgemv.h`` declares, and rejects bad arguments before it
touches the GPU.  No call here reaches a CUDA API, so the suite runs without a
GPU.  Also checks that the product library and the oracle stay separate."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")
PKG = os.path.join(ROOT, "block_quantized_weight_qgemv_gb300")


@pytest.fixture(scope="module")
def qlib():
    from block_quantized_weight_qgemv_gb300 import build
    build.build()
    import block_quantized_weight_qgemv_gb300 as q
    return q


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+char\s*\*|qgemv_status|int64_t|int|void)\s*\**\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["qdequant_q4_0", "qdequant_q4_1", "qdequant_q8_0", "qgemv_q4_0", "qgemv_q4_1",
              "qgemv_q8_0", "qgemm_q4_0", "qgemm_q4_1", "qgemm_q8_0", "qgemv_status_string",
              "qgemv_last_error_string", "qgemv_sync_check", "qgemv_version", "qgemv_shutdown"]:
        assert n in names


def test_library_exports_every_declared_symbol(qlib):
    lib = qlib.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", qlib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported
    # the binding declares a ctypes signature for exactly the header's functions
    assert set(qlib.SIGNATURES) == set(declared_functions())


def test_status_strings_and_version(qlib):
    lib = qlib.lib()
    for code, name in qlib.STATUS.items():
        assert lib.qgemv_status_string(code).decode() == name
    assert lib.qgemv_status_string(99).decode() == "QGEMV_ERR_UNKNOWN"
    assert lib.qgemv_version() >= 100


# Fake, never-dereferenced addresses: validation rejects these calls before
# any CUDA call.
A16 = 0x10000
A8 = 0x10008


def test_gemv_validation_on_host(qlib):
    lib = qlib.lib()
    f = lib.qgemv_q4_0
    assert f(A16, A16, A16, 4, 64, 0, None) == 3          # batch < 1
    assert f(A16, A16, A16, 4, 64, 9, None) == 3          # batch > 8
    assert f(A16, A16, A16, 4, 63, 1, None) == 2          # ncols % 32
    assert f(A16, A16, A16, -1, 64, 1, None) == 2         # negative rows
    assert f(None, A16, A16, 4, 64, 1, None) == 1         # null W
    assert f(A16, None, A16, 4, 64, 1, None) == 1
    assert f(A8, A16, A16, 4, 64, 1, None) == 4           # misaligned W
    assert f(A16, A16, A8, 4, 64, 1, None) == 4           # misaligned y
    assert f(A16, A16, A16, 0, 64, 1, None) == 0          # empty problem: no launch
    assert "batch" in lib.qgemv_last_error_string().decode() or True
    assert lib.qgemv_q8_0(A16, A16, A16, 4, 64, 0, None) == 3
    assert lib.qgemv_q4_1(A16, A16, A16, 4, 40, 1, None) == 2


def test_dequant_and_gemm_validation_on_host(qlib):
    lib = qlib.lib()
    assert lib.qdequant_q4_0(A16, A16, 4, 64, 7, None) == 5     # unknown dtype
    assert lib.qdequant_q4_1(A16, A16, 4, 33, 0, None) == 2
    assert lib.qdequant_q8_0(None, A16, 4, 64, 1, None) == 1
    assert lib.qdequant_q8_0(A16, A8, 4, 64, 1, None) == 4
    assert lib.qdequant_q4_0(A16, A16, 0, 64, 0, None) == 0
    assert lib.qgemm_q4_0(A16, A16, A16, 4, 96, 8, None) == 2   # ncols % 64
    assert lib.qgemm_q4_1(A16, A16, None, 4, 128, 8, None) == 1
    assert lib.qgemm_q8_0(A16, A8, A16, 4, 128, 8, None) == 4
    assert lib.qgemm_q4_0(A16, A16, A16, 4, 128, 0, None) == 0  # m = 0: nothing to do
    msg = lib.qgemv_last_error_string().decode()
    assert msg == ""                                          # cleared by the successful call


def test_mmvq_validation_on_host(qlib):
    lib = qlib.lib()
    assert lib.qgemv_q8_1_size(64, 2) == 160                  # 2*64 codes + 2*2*(4+4) bytes
    assert lib.qgemv_q8_1_size(14336, 1) == 17920
    assert lib.qgemv_q8_1_size(63, 1) == -1
    assert lib.qgemv_q8_1_size(64, 0) == -1
    assert qlib.q8_1_size(4096, 8) == 8 * 4096 * 5 // 4
    for f in (lib.qgemv_mmvq_q4_0, lib.qgemv_mmvq_xq_q4_1, lib.qgemv_mmvq_xq_q8_0):
        assert f(A16, A16, A16, 4, 64, 0, None) == 3          # batch < 1
        assert f(A16, A16, A16, 4, 64, 9, None) == 3          # batch > 8
        assert f(A16, A16, A16, 4, 48, 1, None) == 2          # ncols % 32
        assert f(None, A16, A16, 4, 64, 1, None) == 1
        assert f(A16, None, A16, 4, 64, 1, None) == 1
        assert f(A16, A8, A16, 4, 64, 1, None) == 4           # misaligned x / xq
        assert f(A16, A16, A16, 0, 64, 1, None) == 0          # empty: no launch
    # the one-call form quantizes into a fixed scratch of 2^21 activations
    assert lib.qgemv_mmvq_q8_0(A16, A16, A16, 4, 1 << 19, 8, None) == 2
    assert "scratch" in lib.qgemv_last_error_string().decode()
    assert lib.qquantize_q8_1(A16, A16, 96, 0, None) == 3
    assert lib.qquantize_q8_1(A16, A16, 100, 1, None) == 2
    assert lib.qquantize_q8_1(None, A16, 64, 1, None) == 1
    assert lib.qquantize_q8_1(A16, A8, 64, 1, None) == 4
    assert lib.qquantize_q8_1(A16, A16, 0, 1, None) == 0


def test_gemv_id_validation_on_host(qlib):
    lib = qlib.lib()
    assert qlib.MAX_ID_BATCH == 64
    for f in (lib.qgemv_id_q4_0, lib.qgemv_id_q4_1, lib.qgemv_id_q8_0):
        # (W, n_expert, ids, x, x_group, y, nrows, ncols, batch, stream)
        assert f(A16, 8, A16, A16, 1, A16, 4, 64, 0, None) == 3       # batch < 1
        assert f(A16, 8, A16, A16, 1, A16, 4, 64, 65, None) == 3      # batch > 64
        assert f(A16, 8, A16, A16, 2, A16, 4, 64, 3, None) == 3       # batch not a multiple of x_group
        assert f(A16, 8, A16, A16, 0, A16, 4, 64, 2, None) == 3       # x_group < 1
        assert f(A16, 8, A16, A16, 1, A16, 4, 48, 1, None) == 2       # ncols % 32
        assert f(A16, 0, A16, A16, 1, A16, 4, 64, 1, None) == 2       # no experts
        assert f(A16, 8, A16, A16, 1, A16, -1, 64, 1, None) == 2
        assert f(None, 8, A16, A16, 1, A16, 4, 64, 1, None) == 1
        assert f(A16, 8, None, A16, 1, A16, 4, 64, 1, None) == 1      # null ids
        assert f(A16, 8, A16, A16, 1, None, 4, 64, 1, None) == 1
        assert f(A16, 8, A8, A16, 1, A16, 4, 64, 1, None) == 4        # misaligned ids
        assert f(A16, 8, A16, A8, 1, A16, 4, 64, 1, None) == 4
        assert f(A16, 8, A16, A16, 1, A16, 0, 64, 64, None) == 0      # empty: no launch
    assert lib.qgemv_status_string(11).decode() == "QGEMV_ERR_INDEX"


def test_error_detail_is_recorded(qlib):
    lib = qlib.lib()
    assert lib.qgemv_q4_0(A16, A16, A16, 4, 64, 12, None) == 3
    assert "batch 12" in lib.qgemv_last_error_string().decode()


def test_product_never_touches_the_oracle(qlib):
    """The CUDA library and its binding neither link nor import the oracle."""
    out = subprocess.run(["nm", "-D", qlib.LIB_PATH], capture_output=True, text=True).stdout
    assert "oracle_" not in out
    for dirpath, _, files in os.walk(PKG):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"\boracle\b", src), fn
    hdr = open(HEADER).read()
    assert "oracle" not in hdr
