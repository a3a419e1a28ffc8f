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


@pytest.mark.parametrize("fmt", ["iq3s", "iq2xxs"])
@pytest.mark.parametrize("scale", [2.0 ** -100, 2.0 ** -30, 1.0, 2.0 ** 45, 2.0 ** 110])
@pytest.mark.parametrize("M", [1, 4])
def test_grid_formats_x_range(q, fmt, scale, M):
    """The grid formats on the TMA ring hold each weight as an fp32
    subnormal against x pre-scaled by 2^88; columns whose largest |x| lies
    outside [2^-24, 2^39) are rescaled by a power of two, so every finite x
    meets the tolerance (K = 2048 and 4096: 16-byte rows, the ring)."""
    for N, K in ((70, 2048), (33, 4096)):
        W, tab = synth.gen_cb(fmt, N, K, 600 + N)
        x = (synth.gen_x(M, K, 601) * np.float32(scale)).astype(np.float32)
        Y, A = oracle.gemv_cb(fmt, W, tab, x)
        y = q.qgemv_codebook(fmt, dev(W), dev(tab), dev(x)).cpu().numpy()
        assert np.isfinite(y).all()
        check(y, Y, A, f"{fmt} x scale {scale:g} N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt", ["iq3s", "iq2xxs"])
def test_grid_formats_full_size_sampled(q, fmt):
    """The page-3 grid formats at the IQ3 workload's shape (K=4096,
    N=14336), sampled rows, through the TMA ring."""
    N, K = 14336, 4096
    W, tab = synth.gen_cb(fmt, N, K, 700)
    x = synth.gen_x(1, K, 701)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(5).integers(0, N, 96)]))
    Y, A = oracle.gemv_cb(fmt, W, tab, x, rows=rows)
    y = q.qgemv_codebook(fmt, dev(W), dev(tab), dev(x)).cpu().numpy()
    check(y[:, rows], Y, A, f"{fmt} full size")


@pytest.mark.parametrize("fmt", ["iq3s", "iq2xxs"])
@pytest.mark.parametrize("M", [1, 3])
def test_grid_formats_codebook_bytes_above_127(q, fmt, M):
    """Codebooks with bytes of 128 and more (the published grids stay far
    below) take the expanded table rows: against the oracle, and bit-exact
    through one-hot x."""
    N, K = 70, 2048
    W, tab0 = synth.gen_cb(fmt, N, K, 800)
    rng = np.random.default_rng(801)
    tab = rng.integers(0, 256, tab0.shape, dtype=np.uint8)
    tab.reshape(-1)[0] = 255
    x = synth.gen_x(M, K, 802)
    Y, A = oracle.gemv_cb(fmt, W, tab, x)
    Wg, tg = dev(W), dev(tab)
    check(q.qgemv_codebook(fmt, Wg, tg, dev(x)).cpu().numpy(), Y, A, f"{fmt} codebook bytes >= 128 M={M}")
    Wd = oracle.dequant_cb(fmt, W, tab, K)
    ks = 256 * ((7 * np.arange(32)) % (K // 256)) + 8 * np.arange(32)
    xo = np.zeros((32, K), np.float32)
    xo[np.arange(32), ks] = 1.0
    y = q.qgemv_codebook(fmt, Wg, tg, dev(xo)).cpu().numpy()
    assert np.array_equal(y, Wd[:, ks].T), fmt
