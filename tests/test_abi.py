"""C-ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments on the host (no GPU needed: the pointers below are never
dereferenced because validation fails before any CUDA call)."""
import ctypes
import os
import re

import pytest

from block_quantised_weight_gb300 import build, qgemv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qgemv.load()


def declared_functions():
    txt = open(os.path.join(ROOT, "include", "qgemv.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:QG_API\s+)?(?:const\s+)?\w+\s*\*?\s*(q\w+)\s*\(", txt, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("qgemv_q4k", "qgemv_iq3", "qgemm_q4k_batched", "qdequant_q4k", "qdequant_iq3",
              "qg_device_status", "qg_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) <= set(qgemv.EXPORTS)


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert qgemv.strerror(code) not in ("", "unknown status")
    assert qgemv.strerror(-99) == "unknown status"


A = 0x100000  # fake, 16-byte aligned "device" addresses (never dereferenced)


def _q4k(lib, W, X, Y, M, N, K):
    return lib.qgemv_q4k(W, X, Y, M, N, K, None)


def test_invalid_shapes_rejected_on_host(lib):
    W, X, Y = A, A + 0x10000000, A + 0x20000000
    assert _q4k(lib, W, X, Y, 0, 64, 256) == qgemv.QG_EINVAL
    assert _q4k(lib, W, X, Y, 33, 64, 256) == qgemv.QG_EINVAL
    assert _q4k(lib, W, X, Y, 1, 0, 256) == qgemv.QG_EINVAL
    assert _q4k(lib, W, X, Y, 1, 64, 0) == qgemv.QG_EINVAL
    assert _q4k(lib, W, X, Y, 1, 64, 300) == qgemv.QG_EINVAL
    assert _q4k(lib, None, X, Y, 1, 64, 256) == qgemv.QG_EINVAL
    assert lib.qgemv_iq3(W, None, X, Y, 1, 64, 256, None) == qgemv.QG_EINVAL
    assert lib.qgemm_q4k_batched(W, X, Y, 40, 64, 256, None) == qgemv.QG_EINVAL
    assert lib.qdequant_q4k(W, None, 4, 256, None) == qgemv.QG_EINVAL
    assert lib.qdequant_iq3(W, A + 0x40000000, Y, 4, 257, None) == qgemv.QG_EINVAL


def test_misaligned_pointers_rejected_on_host(lib):
    W, X, Y = A, A + 0x10000000, A + 0x20000000
    assert _q4k(lib, W + 4, X, Y, 1, 64, 256) == qgemv.QG_EALIGN
    assert _q4k(lib, W, X + 8, Y, 1, 64, 256) == qgemv.QG_EALIGN
    assert _q4k(lib, W, X, Y + 4, 1, 64, 256) == qgemv.QG_EALIGN
    assert lib.qgemv_iq3(W, A + 0x30000002, X, Y, 1, 64, 256, None) == qgemv.QG_EALIGN


def test_output_aliasing_rejected_on_host(lib):
    W, X = A, A + 0x10000000
    # Y inside W's 64*144 bytes, then overlapping X
    assert _q4k(lib, W, X, W + 1024, 1, 64, 256) == qgemv.QG_EALIAS
    assert _q4k(lib, W, X, X + 512, 1, 64, 256) == qgemv.QG_EALIAS
    # Y right after X's M*K floats does not overlap: validation passes the
    # alias check (then needs a GPU, so only the codes above are asserted)
    assert lib.qdequant_q4k(W, W + 16, 4, 256, None) == qgemv.QG_EALIAS


def test_group_arguments_rejected_on_host(lib):
    import ctypes
    W = (ctypes.c_void_p * 2)(A, A + 0x1000000)
    Y = (ctypes.c_void_p * 2)(A + 0x2000000, A + 0x3000000)
    N = (ctypes.c_int64 * 2)(64, 64)
    X = A + 0x4000000
    assert lib.qgemv_q4k_group(W, Y, N, 0, X, 1, 256, 0, None) == qgemv.QG_EINVAL
    assert lib.qgemv_q4k_group(W, Y, N, 5, X, 1, 256, 0, None) == qgemv.QG_EINVAL
    assert lib.qgemv_q4k_group(W, Y, N, 2, X, 1, 256, 8, None) == qgemv.QG_EINVAL
    # Y[1] overlapping W[0]
    Y2 = (ctypes.c_void_p * 2)(A + 0x2000000, A + 64)
    assert lib.qgemv_q4k_group(W, Y2, N, 2, X, 1, 256, 0, None) == qgemv.QG_EALIAS
    # Y[0] and Y[1] overlapping each other
    Y3 = (ctypes.c_void_p * 2)(A + 0x2000000, A + 0x2000000 + 128)
    assert lib.qgemv_q4k_group(W, Y3, N, 2, X, 1, 256, 0, None) == qgemv.QG_EALIAS
    assert lib.qgemv_iq3_group(W, Y, N, 2, None, X, 1, 256, 0, None) == qgemv.QG_EINVAL


def test_fused_arguments_rejected_on_host(lib):
    W, X, Y = A, A + 0x10000000, A + 0x20000000
    g, up = A + 0x30000000, A + 0x40000000

    def call(M=1, N=64, K=256, **kw):
        f = qgemv.QgFuse()
        f.norm_weight = kw.get("norm")
        f.norm_eps = kw.get("eps", 1e-5)
        f.up = kw.get("up")
        for i, r in enumerate(kw.get("res", ())):
            f.residual[i] = r
        return lib.qgemv_q4k_fused(W, X, kw.get("Y", Y), M, N, K, ctypes.byref(f), 0, None)

    assert call(norm=g, up=up) == qgemv.QG_EINVAL            # two prologues
    assert call(M=5, norm=g) == qgemv.QG_EINVAL              # prologue needs M <= 4
    assert call(M=5, up=up) == qgemv.QG_EINVAL
    assert call(norm=g, eps=-1.0) == qgemv.QG_EINVAL
    assert call(norm=g, eps=float("nan")) == qgemv.QG_EINVAL
    assert call(norm=g + 4) == qgemv.QG_EALIGN
    assert call(up=up + 8) == qgemv.QG_EALIGN
    assert call(res=(Y + 4,)) == qgemv.QG_EALIGN
    assert call(res=(Y + 16,)) == qgemv.QG_EALIAS             # partial overlap with Y
    assert call(norm=Y + 64) == qgemv.QG_EALIAS
    assert call(res=(None, Y)) == qgemv.QG_EINVAL             # single call: residual[0] only
    Wg = (ctypes.c_void_p * 2)(A, A + 0x1000000)
    Yg = (ctypes.c_void_p * 2)(A + 0x2000000, A + 0x3000000)
    Ng = (ctypes.c_int64 * 2)(64, 64)
    f = qgemv.QgFuse()
    f.residual[0] = A + 0x3000000                             # matrix 0's residual is matrix 1's output
    assert lib.qgemv_q4k_fused_group(Wg, Yg, Ng, 2, X, 1, 256, ctypes.byref(f), 0, None) == qgemv.QG_EALIAS


def test_codebook_arguments_rejected_on_host(lib):
    W, X, Y, B = A, A + 0x10000000, A + 0x20000000, A + 0x30000000
    assert lib.qgemv_codebook(0, W, B, X, Y, 1, 64, 256, None) == qgemv.QG_EINVAL
    assert lib.qgemv_codebook(5, W, B, X, Y, 1, 64, 256, None) == qgemv.QG_EINVAL
    assert lib.qgemv_codebook(1, W, None, X, Y, 1, 64, 256, None) == qgemv.QG_EINVAL
    assert lib.qgemv_codebook(2, W, B + 4, X, Y, 1, 64, 256, None) == qgemv.QG_EALIGN
    assert lib.qgemv_codebook(3, W, B, X, Y, 1, 64, 300, None) == qgemv.QG_EINVAL
    assert lib.qgemv_codebook(4, W, Y + 16, X, Y, 1, 64, 256, None) == qgemv.QG_EALIAS
    assert lib.qdequant_codebook(1, W, B, W + 16, 4, 256, None) == qgemv.QG_EALIAS


def test_chain_step_arguments_rejected_on_host(lib):
    X, Y = A, A + 0x10000000
    assert lib.qg_test_chain_step(None, Y, 2048, 80, 1, None) == qgemv.QG_EINVAL
    assert lib.qg_test_chain_step(X, Y, 300, 80, 1, None) == qgemv.QG_EINVAL
    assert lib.qg_test_chain_step(X, Y, 2048, 0, 1, None) == qgemv.QG_EINVAL
    assert lib.qg_test_chain_step(X, Y, 2048, 80, 4, None) == qgemv.QG_EINVAL
    assert lib.qg_test_chain_step(X + 4, Y, 2048, 80, 1, None) == qgemv.QG_EALIGN
    assert lib.qg_test_chain_step(X, X + 4096, 2048, 80, 1, None) == qgemv.QG_EALIAS
