"""GPU parity of page 3's other codebook formats (qgemv_codebook,
qdequant_codebook: IQ4_NL, IQ4_XS, IQ3_S, IQ2_XXS) against the oracle.

Dequantisation is bit-exact (every value eff * v is exact in fp32); the
GEMV meets |y - y_ref| <= 1e-5 * sum_k |w*x| per element.
"""
import numpy as np
import pytest

import oracle
from block_quantised_weight_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TAU = 1e-5
FORMATS = ["iq4nl", "iq4xs", "iq3s", "iq2xxs"]


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


def check(y, Y, A, what):
    y = np.asarray(y, dtype=np.float64)
    bad = np.abs(y - Y) > TAU * A
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance"


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("N,K", [(1, 256), (33, 512), (7, 2304)])
def test_dequant_bit_exact(q, fmt, N, K):
    W, tab = synth.gen_cb(fmt, N, K, 500 + N + K)
    ref = oracle.dequant_cb(fmt, W, tab, K)
    got = q.qdequant_codebook(fmt, dev(W), dev(tab), K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt", FORMATS)
def test_handworked_blocks_on_gpu(q, golden, fmt):
    from tests.test_oracle_pins import _cb_golden
    W, tab, vals = _cb_golden(golden)[fmt]
    got = q.qdequant_codebook(fmt, dev(W), dev(tab), 256).cpu().numpy()[0]
    for k, v in vals.items():
        assert got[k] == np.float32(v), (fmt, k)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("N,K", [(64, 2048), (100, 768), (257, 4096), (65, 3072), (40, 6144)])
@pytest.mark.parametrize("M", [1, 3, 8, 13, 32])
def test_gemv(q, fmt, N, K, M):
    """IQ4_NL and IQ4_XS rows that are a multiple of 16 bytes take the
    TMA-fed kernel (K = 768, 2048, 3072, 4096, 6144; 768 and 3072 with a
    ragged last chunk of 3 or 4 columns), everything else the direct-load
    kernel."""
    W, tab = synth.gen_cb(fmt, N, K, 600 + N + K)
    x = synth.gen_x(M, K, 601 + M)
    Y, A = oracle.gemv_cb(fmt, W, tab, x)
    y = q.qgemv_codebook(fmt, dev(W), dev(tab), dev(x)).cpu().numpy()
    check(y, Y, A, f"{fmt} N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_gemv_full_size_sampled(q, fmt):
    """The IQ3 config's shape (K=4096, N=14336) in each format, sampled rows."""
    K, N = 4096, 14336
    W, tab = synth.gen_cb(fmt, N, K, 700)
    x = synth.gen_x(1, K, 701)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 48)]))
    Y, A = oracle.gemv_cb(fmt, W, tab, x, rows=rows)
    y = q.qgemv_codebook(fmt, dev(W), dev(tab), dev(x)).cpu().numpy()
    check(y[:, rows], Y, A, f"{fmt} full")
    assert np.isfinite(y).all()


@pytest.mark.parametrize("fmt", FORMATS)
def test_extreme_scales(q, fmt):
    """Every fp16 d field set to an extreme finite value (smallest subnormal,
    smallest normal, 1, 65504), |x| up to 1e3: bit-exact dequantisation and
    the GEMV within tolerance, on the shape each kernel takes (K = 2048)."""
    N, K = 64, 2048
    W, tab = synth.gen_cb(fmt, N, K, 800)
    ext = np.array([0x0001, 0x0400, 0x3C00, 0x7BFF], dtype=np.uint16)
    rng = np.random.default_rng(801)
    step = 18 if fmt == "iq4nl" else synth.CB_UNIT_BYTES[fmt]
    flat = W.reshape(-1, step)
    flat[:, 0:2] = ext[rng.integers(0, 4, len(flat))].view(np.uint8).reshape(-1, 2)
    x = (synth.gen_x(1, K, 802) * 1e3).astype(np.float32)
    ref = oracle.dequant_cb(fmt, W, tab, K)
    got = q.qdequant_codebook(fmt, dev(W), dev(tab), K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    Y, A = oracle.gemv_cb(fmt, W, tab, x)
    y = q.qgemv_codebook(fmt, dev(W), dev(tab), dev(x)).cpu().numpy()
    check(y, Y, A, f"{fmt} extreme scales")
    assert np.isfinite(y).all()
