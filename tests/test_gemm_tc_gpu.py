"""GPU parity of qgemm_q4k_batched against the oracle.

M >= 16 runs the tcgen05 path: Q4_K tiles dequantised and rounded to bf16
(RN), X rounded to bf16, fp32 accumulation.  Each product carries at most
(1 + 2^-9)^2 - 1 < 3.91e-3 relative error, so |y - y_ref| <= 4e-3 * sum|w*x|.
IQ3 keeps its weights exact (signed grid bytes in the MMA, the sub-block
factor applied in fp32 after it), so only the bf16 rounding of X counts
and the same bar holds with room to spare.  M < 16 runs the fp32 FMA path
(1e-5).
"""
import numpy as np
import pytest

import oracle
from block_quantised_weight_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TAU_TC = 4e-3
TAU_FMA = 1e-5


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantised_weight_gb300 import build, qgemv
    build.build()
    qgemv.load()
    return qgemv


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(y, Y, A, tau, what):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - Y)
    bad = err > tau * A
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance; "
                           f"worst ratio {float((err / np.maximum(A, 1e-300)).max()):.3e}")
    return float((err / np.maximum(A, 1e-300)).max())


@pytest.mark.parametrize("N,K,M", [(128, 256, 16), (128, 256, 32), (300, 512, 16), (300, 512, 17),
                                   (1000, 2304, 24), (257, 4096, 32), (64, 768, 31)])
def test_tc_small(q, N, K, M):
    W = synth.gen_q4k(N, K, N + K + M)
    x = synth.gen_x(M, K, M)
    Y, A = oracle.gemv_q4k(W, x)
    y = q.qgemm_q4k_batched(dev(W), dev(x)).cpu().numpy()
    r = check(y, Y, A, TAU_TC, f"tc N={N} K={K} M={M}")
    # the bf16 path is really taken: the error is far above fp32 rounding
    assert r > 1e-6


@pytest.mark.parametrize("M", [1, 2, 8, 15])
def test_batched_below_16_uses_fma_path(q, M):
    N, K = 200, 1024
    W = synth.gen_q4k(N, K, 5)
    x = synth.gen_x(M, K, 6)
    Y, A = oracle.gemv_q4k(W, x)
    check(q.qgemm_q4k_batched(dev(W), dev(x)).cpu().numpy(), Y, A, TAU_FMA, f"batched M={M}")


@pytest.mark.parametrize("K,N,M", [(4096, 11008, 16), (4096, 11008, 32), (8192, 28672, 16), (28672, 8192, 32)])
def test_tc_full_size_sampled(q, K, N, M):
    W = synth.gen_q4k(N, K, K + N)
    x = synth.gen_x(M, K, M + 3)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 64)]))
    Y, A = oracle.gemv_q4k(W, x, rows=rows)
    y = q.qgemm_q4k_batched(dev(W), dev(x)).cpu().numpy()
    check(y[:, rows], Y, A, TAU_TC, f"tc full K={K} N={N} M={M}")
    assert np.isfinite(y).all()
    assert q.qg_device_status() == q.QG_OK


def test_tc_repeatable_within_tolerance(q):
    """Split-K partial sums meet in Y through fp32 atomics: two runs agree to
    rounding, and both meet the tolerance."""
    N, K, M = 512, 8192, 20
    W = dev(synth.gen_q4k(N, K, 9))
    x = dev(synth.gen_x(M, K, 9))
    a = q.qgemm_q4k_batched(W, x).cpu().numpy()
    b = q.qgemm_q4k_batched(W, x).cpu().numpy()
    Y, A = oracle.gemv_q4k(W.cpu().numpy(), x.cpu().numpy())
    check(a, Y, A, TAU_TC, "run a")
    check(b, Y, A, TAU_TC, "run b")
    assert np.allclose(a, b, rtol=0, atol=1e-6 * A.max())


# ------------------------------------------------------------------- IQ3
@pytest.mark.parametrize("N,K,M", [(128, 2048, 16), (300, 2048, 17), (129, 4096, 32), (1000, 2048, 24),
                                   (64, 6144, 31)])
def test_tc_iq3_small(q, N, K, M):
    """IQ3 through tcgen05: every 98-byte block starts 0..14 bytes into its
    112-byte box (all offsets occur for K/256 >= 8)."""
    W, grid = synth.gen_iq3(N, K, N + K + M)
    x = synth.gen_x(M, K, M + 40)
    Y, A = oracle.gemv_iq3(W, grid, x)
    y = q.qgemm_iq3_batched(dev(W), dev(grid), dev(x)).cpu().numpy()
    r = check(y, Y, A, TAU_TC, f"iq3 tc N={N} K={K} M={M}")
    assert r > 1e-6


@pytest.mark.parametrize("M,K", [(8, 2048), (15, 2048), (16, 768), (20, 2304)])
def test_iq3_batched_fma_path(q, M, K):
    """M < 16, or rows not 16-byte aligned (K/256 not a multiple of 8): the
    fp32 FMA path and its 1e-5 bar."""
    N = 150
    W, grid = synth.gen_iq3(N, K, 50 + M)
    x = synth.gen_x(M, K, 51)
    Y, A = oracle.gemv_iq3(W, grid, x)
    check(q.qgemm_iq3_batched(dev(W), dev(grid), dev(x)).cpu().numpy(), Y, A, TAU_FMA, f"iq3 batched M={M}")


@pytest.mark.parametrize("K,N,M", [(8192, 28672, 16), (28672, 8192, 32)])
def test_tc_iq3_full_size_sampled(q, K, N, M):
    W, grid = synth.gen_iq3(N, K, K + N + 1)
    x = synth.gen_x(M, K, M + 5)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 64)]))
    Y, A = oracle.gemv_iq3(W, grid, x, rows=rows)
    y = q.qgemm_iq3_batched(dev(W), dev(grid), dev(x)).cpu().numpy()
    check(y[:, rows], Y, A, TAU_TC, f"iq3 tc full K={K} N={N} M={M}")
    assert np.isfinite(y).all()
    assert q.qg_device_status() == q.QG_OK
