"""Q4_K sub-blocks whose two terms cancel (page 1 "Rewriting picoLM in
Python", dequantize_q4_K: w = d*sc*q - dmin*mn).

A sub-block whose nibbles all equal c, with dmin*mn equal (or nearly equal)
to d*sc*c, has weights that are zero (or tiny) although both terms are
large.  The tolerance is per element, |y - y_ref| <= tau * sum|w*x|, with no
carve-out: a row of such sub-blocks has a tiny sum|w*x| (zero for exact
cancellation, where y must be exactly 0).  Factoring each sub-block as
d*sc * sum(q*x) - dmin*mn * sum(x) loses that accuracy; the kernels factor
around the nearest offset c instead, which keeps it.  Rows of every pattern
below go through the fp32 FMA path (one, four and eight tokens), the
persistent pass kernel and the bf16 tcgen05 path (16 tokens), against the
oracle's fp64 sums.
"""
import numpy as np
import pytest

import oracle
from block_quantised_weight_gb300 import synth

torch = pytest.importorskip("torch")

TAU_FMA, TAU_TC = 1e-5, 4e-3
K = 2048


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


def cancel_block(rng, d, dmin, flips=0, shift=0):
    """One block whose sub-block j has every nibble equal to c_j and
    mn_j = sc_j * c_j + shift (so dmin*mn_j = d*sc_j*c_j when dmin = d and
    shift = 0); `flips` nibbles per sub-block are moved by +-1."""
    sc = np.zeros(8, int)
    mn = np.zeros(8, int)
    c = np.zeros(8, int)
    for j in range(8):
        while True:
            s, cc = int(rng.integers(1, 16)), int(rng.integers(1, 16))
            m = s * cc + shift
            if 0 <= m <= 63:
                break
        sc[j], mn[j], c[j] = s, m, cc
    nib = np.repeat(c[:, None], 32, axis=1)  # [sub-block][l]
    for j in range(8):
        for i in rng.choice(32, size=flips, replace=False):
            nib[j, i] = min(15, max(0, nib[j, i] + (1 if rng.integers(2) else -1)))
    qs = np.zeros(128, np.uint8)
    for g in range(4):   # group g: low nibble -> sub-block 2g, high -> 2g+1
        qs[32 * g:32 * g + 32] = nib[2 * g] | (nib[2 * g + 1] << 4)
    return oracle.q4k_block(d, dmin, sc, mn, qs)


def near_block(rng):
    """A block whose fp16 d, dmin and 6-bit scales are searched so that every
    sub-block's dmin*mn is within 2^-14 (relative), but not equal, to
    d*sc*c; all nibbles of sub-block j equal its c (weights about 2^-14 of
    either term)."""
    S, C, MN = np.meshgrid(np.arange(1, 64), np.arange(1, 16), np.arange(1, 64), indexing="ij")
    while True:
        d = np.float64(np.float16(rng.uniform(1e-3, 4e-3)))
        dmin = np.float64(np.float16(d * rng.uniform(0.3, 3.0)))
        a_c, b = d * S * C, dmin * MN
        rel = np.abs(b - a_c) / a_c
        ok = (rel > 0) & (rel < 2.0 ** -14)
        if ok.sum() >= 8:
            break
    pick = rng.choice(np.flatnonzero(ok), size=8, replace=False)
    sc, c, mn = S.flat[pick], C.flat[pick], MN.flat[pick]
    qs = np.zeros(128, np.uint8)
    for g in range(4):
        qs[32 * g:32 * g + 32] = c[2 * g] | (c[2 * g + 1] << 4)
    return oracle.q4k_block(float(d), float(dmin), sc, mn, qs)


def cancel_rows(seed=0):
    """Rows of several cancellation patterns, plus ordinary random rows."""
    rng = np.random.default_rng(seed)
    one_plus = float(np.float16(1 + 2 ** -10))
    rows, kinds = [], []

    def row(make, kind):
        rows.append(np.concatenate([make() for _ in range(K // 256)]))
        kinds.append(kind)

    for _ in range(6):
        d = float(np.float16(rng.uniform(1e-3, 4e-3)))
        row(lambda: cancel_block(rng, d, d), "exact")                       # w == 0
        row(lambda: cancel_block(rng, -d, -d), "exact, negative scales")    # w == 0
        row(lambda: cancel_block(rng, 1.0, one_plus), "near (2^-10)")       # w = -d*sc*c*2^-10
        row(lambda: cancel_block(rng, d, d, flips=1), "exact + 1 flip")     # w in {0, +-d*sc}
        row(lambda: cancel_block(rng, d, d, flips=3), "exact + 3 flips")
        row(lambda: cancel_block(rng, d, d, shift=1), "off by one min")     # w = -dmin (constant)
        row(lambda: near_block(rng), "near (searched, < 2^-14)")
    W = np.stack(rows)
    W = np.concatenate([W, synth.gen_q4k(8, K, seed + 1)])                  # ordinary rows too
    kinds += ["random"] * 8
    return W, kinds


def check(y, Y, A, tau, kinds, what):
    y = np.asarray(y, dtype=np.float64)
    bad = np.abs(y - Y) > tau * A
    if bad.any():
        m, n = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} outputs out of tolerance; first row {n} ({kinds[n]}), "
                             f"token {m}: y={y[m, n]!r} ref={Y[m, n]!r} A={A[m, n]!r}")


def test_cancellation_rows_are_what_they_claim():
    """The hand-built rows have the intended weights (oracle side, no GPU)."""
    W, kinds = cancel_rows()
    Wd = oracle.dequant_q4k(W, K)
    for n, kind in enumerate(kinds):
        if kind.startswith("exact") and "flip" not in kind:
            assert (Wd[n] == 0).all(), kind
        if kind == "near (2^-10)":
            assert (Wd[n] != 0).all() and np.abs(Wd[n]).max() <= 63 * 2.0 ** -10, kind
        if kind.startswith("near (searched"):
            blk = W[n].reshape(-1, 144)
            d = oracle.f16_to_f32(blk[:, 0:2].copy().view(np.uint16))[:, 0]
            assert (Wd[n] != 0).all()
            # every weight is tiny next to d*sc*q: at most 2^-14 of it
            terms = np.abs(d)[:, None] * 63 * 15
            assert (np.abs(Wd[n].reshape(-1, 256)) <= terms * 2.0 ** -14).all()


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 4, 8])
def test_cancellation_fma_path(q, M):
    W, kinds = cancel_rows()
    x = synth.gen_x(M, K, 7)
    Y, A = oracle.gemv_q4k(W, x)
    assert (A[:, [i for i, k in enumerate(kinds) if k.startswith("exact") and "flip" not in k]] == 0).all()
    y = q.qgemv_q4k(dev(W), dev(x)).cpu().numpy()
    check(y, Y, A, TAU_FMA, kinds, f"FMA path M={M}")


@pytest.mark.gpu
def test_cancellation_pass_kernel(q):
    W, kinds = cancel_rows(3)
    x = synth.gen_x(1, K, 8)
    Y, A = oracle.gemv_q4k(W, x)
    y = torch.empty((1, W.shape[0]), device="cuda")
    sync = torch.zeros(2, dtype=torch.int32, device="cuda")
    q.qgemv_q4k_pass([([dev(W)], [y], dev(x))], sync, M=1)
    check(y.cpu().numpy(), Y, A, TAU_FMA, kinds, "pass kernel")


@pytest.mark.gpu
def test_cancellation_rescaled_x(q):
    """The same rows with x beyond 2^39 (the rescaled decode)."""
    W, kinds = cancel_rows(4)
    x = (synth.gen_x(2, K, 9) * np.float32(2.0 ** 70)).astype(np.float32)
    Y, A = oracle.gemv_q4k(W, x)
    y = q.qgemv_q4k(dev(W), dev(x)).cpu().numpy()
    check(y, Y, A, TAU_FMA, kinds, "rescaled x")


@pytest.mark.gpu
def test_cancellation_tcgen05_path(q):
    """The bf16 path rounds each exact weight once, so it keeps the
    cancellation too: zero weights stay zero and tiny ones keep 2^-9 relative."""
    W, kinds = cancel_rows(5)
    x = synth.gen_x(16, K, 10)
    Y, A = oracle.gemv_q4k(W, x)
    y = q.qgemm_q4k_batched(dev(W), dev(x)).cpu().numpy()
    check(y, Y, A, TAU_TC, kinds, "tcgen05 M=16")
