"""Bit-exact decode inside every GEMV kernel, read out through one-hot x.

With x = e_k (one 1 at position k, zeros elsewhere) each output is a single
dequantised weight, y[n] = w[n][k].  Every kernel forms that value without a
rounding of its own:

* Q4_K (page 1 "Rewriting picoLM in Python", dequantize_q4_K): the min term
  (dmin*mn - d*sc*c) * 1 and the product d*sc * (q - c) are exact and meet in
  one fused multiply-add, the single rounding of d*sc*q - dmin*mn that the
  oracle's fp32 evaluation makes;
* IQ3 in page 4's and page 3's byte orders and page 3's codebook formats:
  products of exact factors (page 3 states that v*eff is exact in fp32);
* the tcgen05 path rounds each weight once to bf16 (RN) and multiplies it by
  x = 1 exactly, so y is the bf16 image of the oracle's value.

So y must equal the oracle's fp32 dequantisation bit for bit (as values: +0
and -0 compare equal), or its bf16 image.  Each launch carries up to 32
one-hot tokens, and the tokens sweep all 256 in-block positions over several
block columns, so every lane position, both halves of a block, every nibble
or index byte and every consumer warp are read out.  x = 2^60 and 2^-100
(outside the directly handled range, so the rescaled path runs) give the
same values times the power of two.
"""
import numpy as np
import pytest

import oracle
from block_quantised_weight_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


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


def positions(K):
    """256 positions, one per in-block offset t, in block (7 t mod K/256)."""
    nb = K // 256
    t = np.arange(256)
    return 256 * ((7 * t) % nb) + t


def onehot(ks, K, value=1.0):
    x = np.zeros((len(ks), K), np.float32)
    x[np.arange(len(ks)), ks] = np.float32(value)
    return x


def expect(Wd, ks, value=1.0):
    """[M, N] expected outputs: w[n][k_m] * value, rounded once to fp32."""
    return (Wd[:, ks].T.astype(np.float64) * value).astype(np.float32)


def bf16_rn(a):
    """fp32 -> the nearest bf16 (ties to even), returned as fp32 (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def sweep(call, Wd, K, group, value=1.0, bf16=False, what=""):
    """Run `call(x)` on the 256 one-hot tokens in launches of `group` tokens."""
    ks = positions(K)
    for s in range(0, 256, group):
        kk = ks[s:s + group]
        y = call(dev(onehot(kk, K, value))).cpu().numpy()
        ref = expect(Wd, kk, value)
        if bf16:
            ref = bf16_rn(ref)
        bad = y != ref
        if bad.any():
            m, n = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: {int(bad.sum())} outputs differ; token k={kk[m]} row {n}: "
                                 f"got {y[m, n]!r} want {ref[m, n]!r}")


# ------------------------------------------------------------ Q4_K, fp32 FMA path
# (N, K) -> launch configuration at one token (launch_q4k.cuh):
#   (70, 4096)    3 tiles x 2 K chunks: split K over 2-CTA clusters
#   (2048, 18432) 64 tiles, 9 chunks: one CTA per SM, deepest ring
#   (9728, 4096)  304 tiles: two CTAs per SM
Q4K_SHAPES = [(70, 4096), (2048, 18432), (9728, 4096)]


@pytest.mark.parametrize("N,K", Q4K_SHAPES)
@pytest.mark.parametrize("group", [1, 6, 32])   # token groups of 1; 6 and 32 (4 x 8) on the tensor cores
def test_onehot_q4k(q, N, K, group):
    W = synth.gen_q4k(N, K, N + K)
    Wd = oracle.dequant_q4k(W, K)
    Wg = dev(W)
    sweep(lambda x: q.qgemv_q4k(Wg, x), Wd, K, group, what=f"q4k N={N} K={K} group={group}")


@pytest.mark.parametrize("value", [2.0 ** 60, 2.0 ** -100])
@pytest.mark.parametrize("group", [1, 4, 8])   # 8: the tensor cores (x in three bf16 parts)
def test_onehot_q4k_rescaled_x(q, value, group):
    """x far outside [2^-24, 2^39): the column is rescaled by 2^-e and its sums by 2^e."""
    N, K = 70, 2048
    W = synth.gen_q4k(N, K, 9)
    Wd = oracle.dequant_q4k(W, K)
    Wg = dev(W)
    sweep(lambda x: q.qgemv_q4k(Wg, x), Wd, K, group, value, what=f"q4k x={value:g} group={group}")


@pytest.mark.parametrize("M", [1, 2, 4])
def test_onehot_q4k_pass_kernel(q, M):
    """The persistent pass kernel (one stage) decodes through the same helpers."""
    N, K = 100, 2048
    W = synth.gen_q4k(N, K, 12)
    Wd = oracle.dequant_q4k(W, K)
    Wg = dev(W)
    sync = torch.zeros(4, dtype=torch.int32, device="cuda")

    def call(x):
        y = torch.empty((x.shape[0], N), device="cuda")
        q.qgemv_q4k_pass([([Wg], [y], x)], sync, M=x.shape[0])
        return y
    sweep(call, Wd, K, M, what=f"pass M={M}")


def test_onehot_q4k_group_launch(q):
    """A grouped launch (q/k/v shapes) with the weight-prefetch flag."""
    K = 2048
    Ws = [synth.gen_q4k(N, K, 20 + N) for N in (300, 64, 64)]
    Wds = [oracle.dequant_q4k(W, K) for W in Ws]
    Wg = [dev(W) for W in Ws]
    for i in range(3):
        sweep(lambda x: q.qgemv_q4k_group(Wg, x, flags=q.QG_PREFETCH_WEIGHTS)[i], Wds[i], K, 4,
              what=f"group matrix {i}")


# ------------------------------------------------------------ IQ3 (both byte orders)
@pytest.mark.parametrize("order", ["page4", "iq3xxs"])
@pytest.mark.parametrize("N,K", [(70, 2048), (130, 4096), (45, 768)])   # K = 768: byte-addressed kernel
@pytest.mark.parametrize("group", [1, 2, 32])   # RG=2 one-token kernel; 2-token; 4-token groups
def test_onehot_iq3(q, order, N, K, group):
    W, grid = synth.gen_iq3(N, K, 3 * N + K)
    if order == "page4":
        Wd = oracle.dequant_iq3(W, grid, K)
        fn = q.qgemv_iq3
    else:
        W = oracle.iq3_to_iq3xxs(W, K)
        Wd = oracle.dequant_iq3xxs(W, grid, K)
        fn = q.qgemv_iq3xxs
    Wg, gg = dev(W), dev(grid)
    sweep(lambda x: fn(Wg, gg, x), Wd, K, group, what=f"iq3 {order} N={N} K={K} group={group}")


@pytest.mark.parametrize("order", ["page4", "iq3xxs"])
@pytest.mark.parametrize("group", [1, 2, 32])
def test_onehot_iq3_grid_bytes_above_127(q, order, group):
    """A grid with bytes of 128 and more (the format allows any byte; the
    published grids stay below 64): each byte lands whole in the low byte
    of its fp32 subnormal."""
    N, K = 70, 2048
    W, _ = synth.gen_iq3(N, K, 11)
    grid = np.random.default_rng(12).integers(0, 256, (256, 4), dtype=np.uint8)
    grid[0, 0] = 255
    if order == "page4":
        Wd = oracle.dequant_iq3(W, grid, K)
        fn = q.qgemv_iq3
    else:
        W = oracle.iq3_to_iq3xxs(W, K)
        Wd = oracle.dequant_iq3xxs(W, grid, K)
        fn = q.qgemv_iq3xxs
    Wg, gg = dev(W), dev(grid)
    sweep(lambda x: fn(Wg, gg, x), Wd, K, group, what=f"iq3 {order} grid bytes >= 128, group={group}")


@pytest.mark.parametrize("value", [2.0 ** 70, 2.0 ** -90])
def test_onehot_iq3_rescaled_x(q, value):
    """x outside [2^-24, 2^39): the IQ3 decode rescales the column."""
    N, K = 70, 2048
    W, grid = synth.gen_iq3(N, K, 5)
    Wd = oracle.dequant_iq3(W, grid, K)
    Wg, gg = dev(W), dev(grid)
    for group in (1, 4):
        sweep(lambda x: q.qgemv_iq3(Wg, gg, x), Wd, K, group, value, what=f"iq3 x={value:g} group={group}")


# ------------------------------------------------------------ page 3 codebook formats
# IQ4_NL and IQ4_XS with 16-byte rows run the TMA-fed kernel; IQ4_XS with an
# odd K/256, IQ3_S and IQ2_XXS the direct-load kernel.
@pytest.mark.parametrize("fmt,K", [("iq4nl", 2048), ("iq4xs", 2048), ("iq4xs", 2304), ("iq3s", 2048),
                                   ("iq2xxs", 2048)])
@pytest.mark.parametrize("group", [1, 32])
def test_onehot_codebook(q, fmt, K, group):
    N = 70
    W, tab = synth.gen_cb(fmt, N, K, 40 + K)
    Wd = oracle.dequant_cb(fmt, W, tab, K)
    Wg, tg = dev(W), dev(tab)
    sweep(lambda x: q.qgemv_codebook(fmt, Wg, tg, x), Wd, K, group, what=f"{fmt} K={K} group={group}")


# ------------------------------------------------------------ tcgen05 (M >= 16)
@pytest.mark.parametrize("fmt", ["q4k", "iq3"])
@pytest.mark.parametrize("group", [16, 32])
def test_onehot_tcgen05_image(q, fmt, group):
    """The tcgen05 path rounds each dequantised Q4_K weight to bf16 (RN)
    once.  IQ3 keeps the signed grid bytes exact in the MMA and applies the
    sub-block factor in fp32 afterwards (their product has at most 24
    significant bits), so a one-hot x returns the weight itself."""
    N, K = 300, 4096
    if fmt == "q4k":
        W = synth.gen_q4k(N, K, 77)
        Wd = oracle.dequant_q4k(W, K)
        Wg = dev(W)
        call = lambda x: q.qgemm_q4k_batched(Wg, x)  # noqa: E731
    else:
        W, grid = synth.gen_iq3(N, K, 78)
        Wd = oracle.dequant_iq3(W, grid, K)
        Wg, gg = dev(W), dev(grid)
        call = lambda x: q.qgemm_iq3_batched(Wg, gg, x)  # noqa: E731
    sweep(call, Wd, K, group, bf16=(fmt == "q4k"), what=f"tcgen05 {fmt} group={group}")
