"""GPU parity: the CUDA path (called through the C ABI) against the CPU oracle.

* qdequant_*: bit-exact (uint32 views equal) with the oracle's fp32 decode.
* qgemv_* (fp32 FMA path): |y - y_ref| <= 1e-5 * sum_k |w*x| per element,
  y_ref and sum|w*x| in fp64 from the oracle; rows with sum|w*x| = 0 exactly 0.
* Full-size shapes of the workloads are checked on sampled rows, in the same
  launch configuration the bench uses.
"""
import numpy as np
import pytest

import oracle
from block_quantised_weight_gb300 import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

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


def check_tol(y, Y, A, tau, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - Y)
    bad = err > tau * A
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first {tuple(i)}: "
                             f"y={y[tuple(i)]!r} ref={Y[tuple(i)]!r} A={A[tuple(i)]!r} "
                             f"ratio={err[tuple(i)] / max(A[tuple(i)], 1e-300):.3e}")
    return float((err / np.maximum(A, 1e-300)).max())


# ------------------------------------------------------------ dequant, exact
@pytest.mark.parametrize("N,K", [(1, 256), (7, 768), (33, 2304), (64, 4096)])
def test_dequant_q4k_bit_exact(q, N, K):
    W = synth.gen_q4k(N, K, 100 + N)
    ref = oracle.dequant_q4k(W, K)
    got = q.qdequant_q4k(dev(W), K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("N,K", [(1, 256), (5, 768), (33, 2304), (40, 4096)])
def test_dequant_iq3_bit_exact(q, N, K):
    W, grid = synth.gen_iq3(N, K, 200 + N)
    ref = oracle.dequant_iq3(W, grid, K)
    got = q.qdequant_iq3(dev(W), dev(grid), K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_handworked_blocks(q, golden):
    # the golden blocks go through the GPU decoder too
    from tests.test_oracle_pins import _iq3_golden, _q4k_golden, _q4k_golden_block
    kv, ws, _ = _q4k_golden(golden)
    blk, _ = _q4k_golden_block(kv, "header")
    got = q.qdequant_q4k(dev(blk), 256).cpu().numpy()[0]
    for i, v in ws:
        assert got[i] == np.float32(v)
    grid, iblk, vals = _iq3_golden(golden)
    goti = q.qdequant_iq3(dev(iblk), dev(grid), 256).cpu().numpy()[0]
    for ib, v in vals.items():
        assert goti[32 * ib:32 * ib + 32].tolist() == v


# ------------------------------------------------------------ GEMV, small
Q4K_SHAPES = [(1, 256), (31, 256), (33, 512), (100, 2304), (64, 2048), (257, 4096), (40, 5632)]


@pytest.mark.parametrize("N,K", Q4K_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8])   # 5-8: the tensor cores, x in three bf16 parts
def test_gemv_q4k_small(q, N, K, M):
    W = synth.gen_q4k(N, K, 7 * N + K)
    x = synth.gen_x(M, K, 3 + M)
    Y, A = oracle.gemv_q4k(W, x)
    y = q.qgemv_q4k(dev(W), dev(x)).cpu().numpy()
    check_tol(y, Y, A, TAU_FMA, f"q4k N={N} K={K} M={M}")


@pytest.mark.parametrize("M", [9, 16, 32])
def test_gemv_q4k_many_tokens(q, M):
    N, K = 70, 1024
    W = synth.gen_q4k(N, K, 5)
    x = synth.gen_x(M, K, 6)
    Y, A = oracle.gemv_q4k(W, x)
    check_tol(q.qgemv_q4k(dev(W), dev(x)).cpu().numpy(), Y, A, TAU_FMA, f"q4k M={M}")


IQ3_SHAPES = [(1, 2048), (31, 2048), (33, 4096), (100, 2048), (70, 6144),
              (5, 256), (33, 768), (40, 2304)]   # the last three: K/256 not a multiple of 8


@pytest.mark.parametrize("N,K", IQ3_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
def test_gemv_iq3_small(q, N, K, M):
    W, grid = synth.gen_iq3(N, K, 11 * N + K)
    x = synth.gen_x(M, K, 4 + M)
    Y, A = oracle.gemv_iq3(W, grid, x)
    y = q.qgemv_iq3(dev(W), dev(grid), dev(x)).cpu().numpy()
    check_tol(y, Y, A, TAU_FMA, f"iq3 N={N} K={K} M={M}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_gemv_iq3_grid_bytes_above_127(q, M):
    """Grid bytes anywhere in 0..255 against the oracle."""
    N, K = 300, 4096
    W, _ = synth.gen_iq3(N, K, 21)
    grid = np.random.default_rng(22).integers(0, 256, (256, 4), dtype=np.uint8)
    x = synth.gen_x(M, K, 23)
    Y, A = oracle.gemv_iq3(W, grid, x)
    y = q.qgemv_iq3(dev(W), dev(grid), dev(x)).cpu().numpy()
    check_tol(y, Y, A, TAU_FMA, f"iq3 grid bytes >= 128 M={M}")


@pytest.mark.parametrize("M", [13, 32])
def test_gemv_iq3_many_tokens(q, M):
    N, K = 45, 2048
    W, grid = synth.gen_iq3(N, K, 8)
    x = synth.gen_x(M, K, 9)
    Y, A = oracle.gemv_iq3(W, grid, x)
    check_tol(q.qgemv_iq3(dev(W), dev(grid), dev(x)).cpu().numpy(), Y, A, TAU_FMA, f"iq3 M={M}")


def test_zero_rows_are_exactly_zero(q):
    N, K = 40, 2048
    W = synth.gen_q4k(N, K, 1)
    W[3] = 0          # d = dmin = 0 everywhere in the row
    W[17, 0:144] = 0  # one zero block inside a live row
    x = synth.gen_x(2, K, 2)
    y = q.qgemv_q4k(dev(W), dev(x)).cpu().numpy()
    assert (y[:, 3] == 0).all()
    Wi, grid = synth.gen_iq3(N, K, 3)
    Wi[5] = 0         # d = 0 everywhere
    yi = q.qgemv_iq3(dev(Wi), dev(grid), dev(x)).cpu().numpy()
    assert (yi[:, 5] == 0).all()


def test_handworked_iq3_gemv(q, golden):
    """The hand-worked IQ3 block dotted with a one-hot x gives its own values."""
    from tests.test_oracle_pins import _iq3_golden
    grid, blk, vals = _iq3_golden(golden)
    W = np.tile(blk, 8)[None, :]              # one row of 8 identical blocks (K = 2048)
    x = np.zeros((4, 2048), np.float32)
    for m, k in enumerate([0, 7, 23, 32 + 5]):
        x[m, k] = 1.0
    y = q.qgemv_iq3(dev(W), dev(grid), dev(x)).cpu().numpy()[:, 0]
    assert y.tolist() == [vals[0][0], vals[0][7], vals[0][23], vals[1][5]]


# ------------------------------------------------------------ full-size shapes
def sampled_rows(N, n=96, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, n)]))


@pytest.mark.parametrize("K,N,M", [(2048, 2048, 1), (4096, 11008, 1), (4096, 11008, 2), (4096, 11008, 4),
                                   (4096, 11008, 8), (8192, 28672, 1), (8192, 28672, 8), (28672, 8192, 1),
                                   (28672, 8192, 8)])
def test_gemv_q4k_full_size_sampled(q, K, N, M):
    W = synth.gen_q4k(N, K, K + N)
    x = synth.gen_x(M, K, M)
    rows = sampled_rows(N)
    Y, A = oracle.gemv_q4k(W, x, rows=rows)
    y = q.qgemv_q4k(dev(W), dev(x)).cpu().numpy()
    check_tol(y[:, rows], Y, A, TAU_FMA, f"q4k full K={K} N={N} M={M}")
    assert np.isfinite(y).all()


@pytest.mark.parametrize("K,N,M", [(4096, 14336, 1), (8192, 28672, 1), (8192, 28672, 8), (28672, 8192, 1),
                                   (28672, 8192, 8)])
def test_gemv_iq3_full_size_sampled(q, K, N, M):
    W, grid = synth.gen_iq3(N, K, K + N + 1)
    x = synth.gen_x(M, K, M + 1)
    rows = sampled_rows(N)
    Y, A = oracle.gemv_iq3(W, grid, x, rows=rows)
    y = q.qgemv_iq3(dev(W), dev(grid), dev(x)).cpu().numpy()
    check_tol(y[:, rows], Y, A, TAU_FMA, f"iq3 full K={K} N={N} M={M}")
    assert np.isfinite(y).all()


def tinyllama_stages():
    """The TinyLlama-shaped decode pass as the bench launches it: q/k/v as one
    group (one x), gate/up as one group, the rest one matrix each; host bytes
    and x per stage."""
    stages = []
    mats = synth.tinyllama_seeds(1)
    i = 0
    while i < len(mats):
        (layer, name, K, N), rng = mats[i]
        take = 3 if name == "q" else 2 if name == "gate" else 1
        Ws, x = [], None
        for j in range(take):
            (_l, nm, Kj, Nj), rj = mats[i + j]
            Ws.append((f"{layer}.{nm}", synth.gen_q4k(Nj, Kj, rj)))
            xj = synth.gen_x(1, Kj, rj)
            x = xj if x is None else x   # the group shares the first matrix's x
        stages.append((layer, Ws, x))
        i += take
    assert len(stages) == 89
    return stages


def test_tinyllama_pass_sampled(q):
    """Every one of the 155 matrices of the TinyLlama-shaped decode pass,
    sampled rows against the oracle, through the entry point and flag the
    bench times (qgemv_q4k_group with QG_PREFETCH_WEIGHTS; q/k/v and gate/up
    grouped)."""
    for layer, Ws, x in tinyllama_stages():
        ys = q.qgemv_q4k_group([dev(W) for _n, W in Ws], dev(x), flags=q.QG_PREFETCH_WEIGHTS)
        for (name, W), y in zip(Ws, ys):
            rows = sampled_rows(W.shape[0], 24, seed=layer)
            Y, A = oracle.gemv_q4k(W, x, rows=rows)
            check_tol(y.cpu().numpy()[:, rows], Y, A, TAU_FMA, f"tinyllama {name}")
    assert q.qg_device_status() == q.QG_OK


# ------------------------------------------------------------ errors
def test_bounded_wait_reports_timeout_and_context_survives(q):
    assert q.qg_device_status() == q.QG_OK
    assert q.qg_test_bounded_wait() == q.QG_OK
    assert q.qg_device_status() == q.QG_ETIMEOUT
    assert q.qg_device_status() == q.QG_OK   # cleared
    W = synth.gen_q4k(8, 512, 0)
    x = synth.gen_x(1, 512, 0)
    Y, A = oracle.gemv_q4k(W, x)
    check_tol(q.qgemv_q4k(dev(W), dev(x)).cpu().numpy(), Y, A, TAU_FMA, "after timeout")


def test_binding_raises_on_bad_arguments(q):
    W = dev(synth.gen_q4k(4, 512, 0))
    x = torch.zeros((33, 512), device="cuda")
    with pytest.raises(q.QGError) as e:
        q.qgemv_q4k(W, x)
    assert e.value.code == q.QG_EINVAL
    with pytest.raises(TypeError):
        q.qgemv_q4k(W.cpu(), x[:1])
    y = torch.empty((1, 4), device="cuda")
    rc = q.load().qgemv_q4k(W.data_ptr() + 4, x.data_ptr(), y.data_ptr(), 1, 4, 512, None)
    assert rc == q.QG_EALIGN


# ------------------------------------------------------------ dependent launch
@pytest.mark.parametrize("fmt,M", [("q4k", 1), ("iq3", 1), ("q4k", 4), ("q4k", 8)])   # q4k 8: tensor cores
def test_prefetch_flag_dependency_chain(q, fmt, M):
    """x_{i+1} = y_i through six square GEMVs issued back to back on one stream.
    With QG_PREFETCH_WEIGHTS each launch may start before its predecessor ends;
    the results must equal the plain stream-ordered launches bit for bit and
    match the oracle stage by stage.  From 5 tokens the tensor-core path runs
    (the flag changes nothing there) and its split rows meet in fp32 atomics,
    so the two chains agree to the order of those additions."""
    K = N = 2048
    mats = []
    for i in range(6):
        if fmt == "q4k":
            mats.append((dev(synth.gen_q4k(N, K, 300 + i)), None))
        else:
            W, grid = synth.gen_iq3(N, K, 400 + i)
            mats.append((dev(W), dev(grid)))
    x0 = dev(synth.gen_x(M, K, 7))

    def chain(flags):
        xs = [x0]
        for W, g in mats:
            if fmt == "q4k":
                y = q.qgemv_q4k(W, xs[-1], flags=flags)
            else:
                y = q.qgemv_iq3(W, g, xs[-1], flags=flags)
            xs.append(y / 32.0)   # keep magnitudes bounded (exact scaling)
        torch.cuda.synchronize()
        return xs

    plain = chain(0)
    fast = chain(q.QG_PREFETCH_WEIGHTS)
    for a, b in zip(plain, fast):
        if M >= 5:
            assert torch.allclose(a, b, rtol=0, atol=1e-6 * float(a.abs().max()))
        else:
            assert torch.equal(a, b)
    # each stage on the oracle's own chain of inputs (fp32 of the oracle's
    # previous output / 32), with and without the flag
    xin = x0.cpu().numpy().reshape(M, K)
    for i, (W, g) in enumerate(mats):
        Wh = W.cpu().numpy()
        if fmt == "q4k":
            Y, A = oracle.gemv_q4k(Wh, xin)
            ys = [q.qgemv_q4k(W, dev(xin), flags=f) for f in (0, q.QG_PREFETCH_WEIGHTS)]
        else:
            Y, A = oracle.gemv_iq3(Wh, g.cpu().numpy(), xin)
            ys = [q.qgemv_iq3(W, g, dev(xin), flags=f) for f in (0, q.QG_PREFETCH_WEIGHTS)]
        for y in ys:
            check_tol(y.cpu().numpy(), Y, A, TAU_FMA, f"chain stage {i}")
        xin = (Y / 32.0).astype(np.float32)
    assert q.qg_device_status() == q.QG_OK


def test_prefetch_flag_rejects_unknown_bits(q):
    W = dev(synth.gen_q4k(4, 512, 0))
    x = torch.zeros((1, 512), device="cuda")
    y = torch.empty((1, 4), device="cuda")
    assert q.load().qgemv_q4k_ex(W.data_ptr(), x.data_ptr(), y.data_ptr(), 1, 4, 512, 6, None) == q.QG_EINVAL


# ------------------------------------------------------------ grouped launches
@pytest.mark.parametrize("M", [1, 3, 9])
def test_q4k_group_matches_single_calls(q, M):
    """q, k, v of one TinyLlama layer (2048x2048, 256x2048, 256x2048) in one
    launch, reading the same x: identical to three separate launches (from 5
    tokens, the tensor-core path, up to the order of its fp32 atomics)."""
    K = 2048
    Ws = [dev(synth.gen_q4k(N, K, 50 + N + i)) for i, N in enumerate((2048, 256, 256))]
    x = dev(synth.gen_x(M, K, 11))
    ys = q.qgemv_q4k_group(Ws, x)
    for W, y in zip(Ws, ys):
        r = q.qgemv_q4k(W, x)
        if M >= 5:
            assert torch.allclose(y, r, rtol=0, atol=1e-6 * float(r.abs().max()))
        else:
            assert torch.equal(y, r)
        Y, A = oracle.gemv_q4k(W.cpu().numpy(), x.cpu().numpy(), rows=np.arange(0, W.numel() // 1152, 7))
        check_tol(y.cpu().numpy()[:, ::7], Y, A, TAU_FMA, "group")


def test_q4k_group_with_prefetch_flag(q):
    K = 2048
    Ws = [dev(synth.gen_q4k(N, K, 70 + i)) for i, N in enumerate((5632, 5632))]
    x = dev(synth.gen_x(1, K, 12))
    a = q.qgemv_q4k_group(Ws, x, flags=q.QG_PREFETCH_WEIGHTS)
    b = [q.qgemv_q4k(W, x) for W in Ws]
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.parametrize("K", [2048, 768])
@pytest.mark.parametrize("M", [1, 2, 4, 5])
def test_iq3_group_matches_single_calls(q, K, M):
    """Bit-identical on the FMA paths; from 5 tokens with K/256 a multiple
    of 8 (the tensor-core path) split rows meet in fp32 atomics, so the two
    agree to the order of those additions."""
    grid = synth.gen_iq3_grid(3)
    Ws = [dev(synth.gen_iq3(N, K, 80 + i, grid_seed=3)[0]) for i, N in enumerate((100, 64, 33))]
    g = dev(grid)
    x = dev(synth.gen_x(M, K, 13))
    ys = q.qgemv_iq3_group(Ws, g, x)
    for W, y in zip(Ws, ys):
        r = q.qgemv_iq3(W, g, x)
        if M >= 5 and (K // 256) % 8 == 0:
            assert torch.allclose(y, r, rtol=0, atol=1e-6 * float(r.abs().max()))
        else:
            assert torch.equal(y, r)


# ------------------------------------------------------------ persistent pass
@pytest.mark.parametrize("M", [1, 2])
def test_pass_kernel_dependent_stages(q, M):
    """Stages whose X is the previous stage's Y, in one persistent launch:
    identical to launching the groups one by one, and matching the oracle
    stage by stage."""
    rng = np.random.default_rng(40 + M)

    def W(N, K):
        return dev(synth.gen_q4k(N, K, rng))

    x0 = dev(synth.gen_x(M, 512, 5))
    A, B = W(512, 512), W(256, 512)
    C = W(768, 512)
    D = W(256, 768)
    E, F = W(100, 256), W(64, 256)
    yA, yB = torch.empty((M, 512), device="cuda"), torch.empty((M, 256), device="cuda")
    yC = torch.empty((M, 768), device="cuda")
    yD = torch.empty((M, 256), device="cuda")
    yE, yF = torch.empty((M, 100), device="cuda"), torch.empty((M, 64), device="cuda")
    stages = [([A, B], [yA, yB], x0), ([C], [yC], yA), ([D], [yD], yC), ([E, F], [yE, yF], yD)]
    sync = torch.zeros(8, dtype=torch.int32, device="cuda")
    for _ in range(2):   # twice: the sync words are re-zeroed by each call
        for ys in (yA, yB, yC, yD, yE, yF):
            ys.fill_(float("nan"))
        q.qgemv_q4k_pass(stages, sync, M=M)
        torch.cuda.synchronize()
        ref = []
        for Ws, Ys, X in stages:
            ref.append(q.qgemv_q4k_group(Ws, X))
        torch.cuda.synchronize()
        for (Ws, Ys, X), r in zip(stages, ref):
            for y, yr in zip(Ys, r):
                assert torch.equal(y, yr)
    # the same stages on the oracle's own chain of inputs (fp32 of the
    # oracle's yA, yC, yD), each in its own buffer: the pass still orders
    # the stages, and every output meets the oracle
    host = {id(W): W.cpu().numpy() for Ws, _, _ in stages for W in Ws}
    xo = [x0.cpu().numpy()]
    for W in (A, C, D):
        xo.append(oracle.gemv_q4k(host[id(W)], xo[-1])[0].astype(np.float32))
    indep = [(Ws, [torch.empty_like(y) for y in Ys], dev(x)) for (Ws, Ys, _), x in zip(stages, xo)]
    q.qgemv_q4k_pass(indep, sync, M=M)
    for (Ws, Ys, _), x in zip(indep, xo):
        for Wt, y in zip(Ws, Ys):
            Y, Aa = oracle.gemv_q4k(host[id(Wt)], x)
            check_tol(y.cpu().numpy(), Y, Aa, TAU_FMA, "pass stage")
    assert q.qg_device_status() == q.QG_OK


def test_tinyllama_pass_kernel_matches_groups(q):
    """The 89-stage TinyLlama pass (q/k/v and gate/up grouped) as one
    persistent launch: sampled rows of every stage against the oracle, and
    equal bit for bit to the stage-by-stage grouped launches where both add
    the K chunks in the same order (one chunk, K = 2048; the grouped launch
    splits K = 5632 over a cluster and sums its three chunks in another
    order, so there each is held to the oracle on its own)."""
    host = tinyllama_stages()
    stages = []
    for _layer, Ws, x in host:
        Wd = [dev(W) for _n, W in Ws]
        stages.append((Wd, [torch.empty((1, W.shape[0]), device="cuda") for _n, W in Ws], dev(x)))
    sync = torch.zeros(89, dtype=torch.int32, device="cuda")
    q.qgemv_q4k_pass(stages, sync, M=1)
    for (layer, Ws, x), (Wd, Ys, X) in zip(host, stages):
        K = x.shape[-1]
        grouped = q.qgemv_q4k_group(Wd, X)
        for (name, W), y, yr in zip(Ws, Ys, grouped):
            if K <= 2048:
                assert torch.equal(y, yr), name
            rows = sampled_rows(W.shape[0], 24, seed=layer)
            Y, A = oracle.gemv_q4k(W, x, rows=rows)
            check_tol(y.cpu().numpy()[:, rows], Y, A, TAU_FMA, f"pass {name}")
            check_tol(yr.cpu().numpy()[:, rows], Y, A, TAU_FMA, f"grouped {name}")
    assert q.qg_device_status() == q.QG_OK


# Token scales from 2^-100 to 2^110 (gen_x draws |x| < 5): with the synthetic
# scales the outputs stay normal fp32 numbers, whose own rounding is then far
# inside the tolerance.  Subnormal x is covered with large block scales below.
X_SCALES = [2.0 ** -100, 2.0 ** -80, 2.0 ** -30, 1.0, 2.0 ** 38, 2.0 ** 60, 2.0 ** 110]


def big_scales(W, block_bytes, d_off, dmin_off=None, seed=0):
    """Set every block's fp16 d (and dmin) to values in [2^14, 2^15), so that
    x near 2^-140 still gives outputs that are normal fp32 numbers."""
    rng = np.random.default_rng(seed)
    blk = W.reshape(-1, block_bytes)
    for off in (d_off, dmin_off):
        if off is not None:
            v = (rng.uniform(2 ** 14, 2 ** 15, len(blk))).astype(np.float16)
            blk[:, off:off + 2] = v.view(np.uint8).reshape(-1, 2)
    return W


@pytest.mark.parametrize("scale", X_SCALES)
@pytest.mark.parametrize("M", [1, 4])
def test_gemv_q4k_x_range(q, scale, M):
    """The Q4_K decode holds each nibble as an fp32 subnormal against x
    pre-scaled by 2^76..2^88; a slice whose largest |x| falls outside
    [2^-24, 2^39) is first rescaled by a power of two (undone on its partial
    sums), so every finite x meets the fp32 tolerance."""
    N, K = 96, 2048
    W = synth.gen_q4k(N, K, 31)
    x = (synth.gen_x(M, K, 32) * np.float32(scale)).astype(np.float32)
    Y, A = oracle.gemv_q4k(W, x)
    y = q.qgemv_q4k(dev(W), dev(x)).cpu().numpy()
    assert np.isfinite(y).all()
    check_tol(y, Y, A, TAU_FMA, f"x scale {scale:g}, M={M}")


@pytest.mark.parametrize("scale", [2.0 ** -100, 2.0 ** -60, 1.0, 2.0 ** 60, 2.0 ** 100])
@pytest.mark.parametrize("fmt", ["q4k", "iq3"])
def test_gemv_x_range_tensor_cores(q, fmt, scale):
    """From 5 tokens both formats run on the tensor cores with x split into
    three bf16 parts and multiplied as given: the stated range |x| within
    [2^-100, 2^100] meets the fp32 bar."""
    N, K, M = 96, 2048, 8
    x = (synth.gen_x(M, K, 40) * np.float32(scale)).astype(np.float32)
    if fmt == "q4k":
        W = synth.gen_q4k(N, K, 41)
        Y, A = oracle.gemv_q4k(W, x)
        y = q.qgemv_q4k(dev(W), dev(x)).cpu().numpy()
    else:
        W, grid = synth.gen_iq3(N, K, 42)
        Y, A = oracle.gemv_iq3(W, grid, x)
        y = q.qgemv_iq3(dev(W), dev(grid), dev(x)).cpu().numpy()
    assert np.isfinite(y).all()
    check_tol(y, Y, A, TAU_FMA, f"{fmt} tensor cores x scale {scale:g}")


@pytest.mark.parametrize("M", [1, 4])
def test_gemv_subnormal_x(q, M):
    """x entirely subnormal (|x| < 2^-137) against blocks with d near 2^15:
    both FMA decodes rescale it by 2^100 and meet the tolerance."""
    N, K = 96, 2048
    x = (synth.gen_x(M, K, 37) * np.float32(2.0 ** -140)).astype(np.float32)
    assert (np.abs(x) < 2.0 ** -126).all()
    W = big_scales(synth.gen_q4k(N, K, 38), 144, 0, 2)
    Y, A = oracle.gemv_q4k(W, x)
    assert (np.abs(Y) > 2.0 ** -120).mean() > 0.9
    check_tol(q.qgemv_q4k(dev(W), dev(x)).cpu().numpy(), Y, A, TAU_FMA, f"q4k subnormal x M={M}")
    Wi, grid = synth.gen_iq3(N, K, 39)
    Wi = big_scales(Wi, 98, 96)
    Y, A = oracle.gemv_iq3(Wi, grid, x)
    check_tol(q.qgemv_iq3(dev(Wi), dev(grid), dev(x)).cpu().numpy(), Y, A, TAU_FMA, f"iq3 subnormal x M={M}")


def test_gemv_q4k_x_mixed_ranges(q):
    """One launch whose tokens, and whose columns within a row, mix the
    directly handled range with rescaled ones (per-column, per-token
    exponents), through the one-token, four-token and cluster launches."""
    for N, K in ((96, 2048), (70, 4096), (700, 4096)):
        W = synth.gen_q4k(N, K, 33)
        x = synth.gen_x(4, K, 34)
        x[0] *= np.float32(2.0 ** 100)
        x[1, : K // 2] *= np.float32(2.0 ** -60)      # half the columns tiny
        x[2, K // 2:] *= np.float32(2.0 ** 80)       # half the columns huge
        x[3, 256:512] *= np.float32(2.0 ** 45)       # one column just above the direct range
        Y, A = oracle.gemv_q4k(W, x)
        for M in (1, 4):
            y = q.qgemv_q4k(dev(W), dev(x[:M] if M == 4 else x[3:4])).cpu().numpy()
            Ys, As = (Y, A) if M == 4 else (Y[3:4], A[3:4])
            check_tol(y, Ys, As, TAU_FMA, f"mixed ranges N={N} K={K} M={M}")


@pytest.mark.parametrize("scale", X_SCALES)
@pytest.mark.parametrize("M", [1, 2, 4])
def test_gemv_iq3_x_range(q, scale, M):
    """The IQ3 decode takes columns whose largest |x| is in [2^-24, 2^39) as
    they are (x pre-scaled by 2^88 against grid bytes held as fp32
    subnormals) and rescales the others by a power of two."""
    N, K = 96, 2048
    W, grid = synth.gen_iq3(N, K, 35)
    x = (synth.gen_x(M, K, 36) * np.float32(scale)).astype(np.float32)
    Y, A = oracle.gemv_iq3(W, grid, x)
    y = q.qgemv_iq3(dev(W), dev(grid), dev(x)).cpu().numpy()
    assert np.isfinite(y).all()
    check_tol(y, Y, A, TAU_FMA, f"iq3 x scale {scale:g}, M={M}")


# ------------------------------------------------------------ IQ3_XXS (page 3 order)
@pytest.mark.parametrize("N,K", [(1, 256), (33, 2304), (40, 4096)])
def test_dequant_iq3xxs_bit_exact(q, N, K):
    W, grid = synth.gen_iq3(N, K, 300 + N)
    W = oracle.iq3_to_iq3xxs(W, K)
    ref = oracle.dequant_iq3xxs(W, grid, K)
    got = q.qdequant_iq3xxs(dev(W), dev(grid), K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_iq3xxs_handworked_block(q, golden):
    from tests.test_oracle_pins import _iq3xxs_golden
    grid, blk, vals = _iq3xxs_golden(golden)
    got = q.qdequant_iq3xxs(dev(blk), dev(grid), 256).cpu().numpy()[0]
    for ib, v in vals.items():
        assert got[32 * ib:32 * ib + 32].tolist() == v


@pytest.mark.parametrize("N,K", [(64, 2048), (100, 4096), (300, 2048), (33, 768), (57, 6144)])
@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_gemv_iq3xxs(q, N, K, M):
    """Both decode paths (two-row half blocks for M <= 2, whole blocks for
    M > 2) and the byte-addressed path (K/256 not a multiple of 8)."""
    W, grid = synth.gen_iq3(N, K, 400 + N + K)
    W = oracle.iq3_to_iq3xxs(W, K)
    x = synth.gen_x(M, K, 401)
    Y, A = oracle.gemv_iq3xxs(W, grid, x)
    y = q.qgemv_iq3xxs(dev(W), dev(grid), dev(x)).cpu().numpy()
    check_tol(y, Y, A, TAU_FMA, f"iq3xxs N={N} K={K} M={M}")


def test_gemv_iq3xxs_full_size_sampled(q):
    K, N = 8192, 28672
    W, grid = synth.gen_iq3(N, K, 4)
    W = oracle.iq3_to_iq3xxs(W, K)
    x = synth.gen_x(1, K, 5)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 64)]))
    Y, A = oracle.gemv_iq3xxs(W, grid, x, rows=rows)
    y = q.qgemv_iq3xxs(dev(W), dev(grid), dev(x), flags=q.QG_PREFETCH_WEIGHTS).cpu().numpy()
    check_tol(y[:, rows], Y, A, TAU_FMA, "iq3xxs full")


def _probe_value(x):
    """What one CTA of the probe writes: warp 0's share of sum(x), thread t
    taking float4 groups t, t + 288, ... (288 threads per CTA)."""
    g = x.double().reshape(-1, 4).sum(1)
    return float(sum(g[t::288].sum() for t in range(32)))


def test_chain_step_probe(q):
    """qg_test_chain_step (the dependent-launch floor probe): every CTA writes
    the same value (its first warp's share of sum(x)) into its 32 outputs,
    with and without the programmatic dependent launch flag, in a chain that
    reads the previous launch's output."""
    import ctypes
    lib = q.load()
    K, grid = 2048, 80
    x = torch.arange(K, dtype=torch.float32, device="cuda") / K
    y = torch.zeros(grid * 32, dtype=torch.float32, device="cuda")
    y2 = torch.zeros(grid * 32, dtype=torch.float32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for flags in (0, q.QG_PREFETCH_WEIGHTS):
        assert lib.qg_test_chain_step(x.data_ptr(), y.data_ptr(), K, grid, flags, s) == 0
        assert lib.qg_test_chain_step(y.data_ptr(), y2.data_ptr(), K, grid, flags, s) == 0
        torch.cuda.synchronize()
        assert torch.allclose(y.double(), torch.full_like(y.double(), _probe_value(x)), rtol=1e-5)
        assert torch.allclose(y2.double(), torch.full_like(y2.double(), _probe_value(y[:K])), rtol=1e-5)


def test_concurrent_host_threads(q):
    """Eight host threads calling four entry points at once, each on its own
    stream (the binding releases the GIL for the C call), get the results of
    the same calls made one at a time.  A thread whose first CUDA call is the
    library's must work too: the tensor-map encoder is a driver call that
    needs the runtime's context bound to the thread."""
    import threading
    K, N = 2048, 300
    Wq = dev(synth.gen_q4k(N, K, 11))
    Wi_np, grid_np = synth.gen_iq3(N, K, 12)
    Wi, grid = dev(Wi_np), dev(grid_np)
    Wc_np, tab_np = synth.gen_cb("iq4nl", N, K, 13)
    Wc, tab = dev(Wc_np), dev(tab_np)
    x1 = dev(synth.gen_x(1, K, 14))
    x16 = dev(synth.gen_x(16, K, 15))
    calls = [lambda s: q.qgemv_q4k(Wq, x1, stream=s),
             lambda s: q.qgemv_iq3(Wi, grid, x1, stream=s),
             lambda s: q.qgemv_codebook("iq4nl", Wc, tab, x1, stream=s),
             lambda s: q.qgemm_q4k_batched(Wq, x16, stream=s)]
    ref = []
    for c in calls:
        ref.append(c(None).cpu())
    torch.cuda.synchronize()
    outs, errs = [None] * 8, []

    def run(i):
        try:
            s = torch.cuda.Stream()
            y = calls[i % 4](s)
            s.synchronize()
            outs[i] = y.cpu()
        except Exception as e:  # reported below
            errs.append(e)

    ts = [threading.Thread(target=run, args=(i,)) for i in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    for i, y in enumerate(outs):
        r = ref[i % 4]
        if i % 4 == 3:  # tcgen05 path: split tiles meet in fp32 atomics, summation order varies
            assert torch.allclose(y, r, rtol=1e-5, atol=1e-6 * float(r.abs().max())), i
        else:           # FMA paths: deterministic
            assert torch.equal(y, r), i
    assert q.qg_device_status() == 0


# fp16 scale fields at the ends of their range: the smallest subnormal, the
# smallest normal, 1, and the largest finite value (65504).
_EXTREME_F16 = np.array([0x0001, 0x0400, 0x3C00, 0x7BFF], dtype=np.uint16)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_q4k_extreme_scales(q, M):
    """Q4_K blocks whose d and dmin take the extreme finite fp16 values, with
    |x| up to 1e3: dequantisation stays bit-exact and the GEMV (including the
    x pre-scaling by 2^76..2^88 of the nibble trick, and the tcgen05 path at
    M = 16) within its tolerance."""
    N, K = 96, 1024
    W = synth.gen_q4k(N, K, 31)
    blk = W.reshape(-1, 144)
    rng = np.random.default_rng(32)
    blk[:, 0:2] = _EXTREME_F16[rng.integers(0, 4, len(blk))].view(np.uint8).reshape(-1, 2)
    blk[:, 2:4] = _EXTREME_F16[rng.integers(0, 4, len(blk))].view(np.uint8).reshape(-1, 2)
    x = (synth.gen_x(M, K, 33) * 1e3).astype(np.float32)
    ref = oracle.dequant_q4k(W, K)
    got = q.qdequant_q4k(dev(W), K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    Y, A = oracle.gemv_q4k(W, x)
    y = q.qgemm_q4k_batched(dev(W), dev(x)).cpu().numpy()
    check_tol(y, Y, A, 4e-3 if M >= 16 else TAU_FMA, f"q4k extreme scales M={M}")
    assert np.isfinite(y).all()


@pytest.mark.parametrize("M", [1, 2, 16])
def test_iq3_extreme_scales(q, M):
    """IQ3 super-blocks whose d takes the extreme finite fp16 values, |x| up
    to 1e3: bit-exact dequantisation, GEMV within tolerance (FMA path, and
    the tcgen05 path at M = 16)."""
    N, K = 96, 2048
    W, grid = synth.gen_iq3(N, K, 41)
    blk = W.reshape(-1, 98)
    rng = np.random.default_rng(42)
    blk[:, 96:98] = _EXTREME_F16[rng.integers(0, 4, len(blk))].view(np.uint8).reshape(-1, 2)
    x = (synth.gen_x(M, K, 43) * 1e3).astype(np.float32)
    ref = oracle.dequant_iq3(W, grid, K)
    got = q.qdequant_iq3(dev(W), dev(grid), K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    Y, A = oracle.gemv_iq3(W, grid, x)
    y = q.qgemm_iq3_batched(dev(W), dev(grid), dev(x)).cpu().numpy()
    check_tol(y, Y, A, 4e-3 if M >= 16 else TAU_FMA, f"iq3 extreme scales M={M}")
    assert np.isfinite(y).all()
