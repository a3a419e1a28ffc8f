"""GPU parity of the fused decode-step GEMVs (qgemv_q4k_fused / _group)
against the fp64 oracle: RMSNorm or SwiGLU prologue on x, residual epilogue.

Bar: |y - y_ref| <= 1e-5 * sum_k |w*h| (h the exact prologue output) plus
2^-23 * |y_ref| for the fp32 residual add, per element.  Shapes span one
and several K chunks (2048 columns each), a ragged last chunk, the
split-K cluster launch (M=1, few tiles, several chunks) and ragged N.
"""
import numpy as np
import pytest

import oracle
from block_quantised_weight_gb300 import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TAU = 1e-5


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


def check(y, Y, A, res=False, what=""):
    y = np.asarray(y, dtype=np.float64).reshape(Y.shape)
    tol = TAU * A + (2.0 ** -23 * np.abs(Y) if res else 0.0)
    bad = np.abs(y - Y) > tol
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} out of tolerance; first {i}: y={y[i]!r} ref={Y[i]!r} A={A[i]!r}")


SHAPES = [(77, 512), (64, 2048), (300, 2304), (64, 5632), (33, 6144)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_rmsnorm_prologue(q, N, K, M):
    W = synth.gen_q4k(N, K, 1000 + N + K)
    x = synth.gen_x(M, K, 7 + M)
    g = synth.gen_x(1, K, 8)[0]
    Y, A = oracle.fused_gemv_q4k(W, x, norm_weight=g, eps=1e-5)
    y = q.qgemv_q4k_fused(dev(W), dev(x), norm_weight=dev(g), eps=1e-5)
    check(y.cpu().numpy(), Y, A, what=f"rmsnorm M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 4])
def test_swiglu_prologue_with_residual(q, N, K, M):
    W = synth.gen_q4k(N, K, 2000 + N + K)
    gate = 3.0 * synth.gen_x(M, K, 9)
    up = synth.gen_x(M, K, 10)
    R = synth.gen_x(M, N, 11)
    Y, A = oracle.fused_gemv_q4k(W, gate, up=up, residual=R)
    y = q.qgemv_q4k_fused(dev(W), dev(gate), up=dev(up), residual=dev(R))
    check(y.cpu().numpy(), Y, A, res=True, what=f"swiglu M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(77, 512), (64, 5632), (2048, 2048)])
def test_residual_in_place(q, N, K):
    """residual == out: Y += X W^T (the o and down projections' skip adds)."""
    W = synth.gen_q4k(N, K, 3000 + N)
    x = synth.gen_x(1, K, 12)
    R = synth.gen_x(1, N, 13)
    Y, A = oracle.fused_gemv_q4k(W, x, residual=R)
    out = dev(R.copy())
    q.qgemv_q4k_fused(dev(W), dev(x), out=out, residual=out)
    check(out.cpu().numpy(), Y, A, res=True, what="in-place residual")


def test_large_activations_and_extreme_silu(q):
    """Gate values far into both tails (exp(-z) overflows to inf, silu -> 0)
    and an RMSNorm input of large magnitude (the 1/rms scale is applied after
    the dot product)."""
    K, N = 2048, 96
    W = synth.gen_q4k(N, K, 4000)
    gate = synth.gen_x(1, K, 14) * 60.0
    gate[0, :16] = -200.0
    gate[0, 16:32] = 200.0
    up = synth.gen_x(1, K, 15)
    Y, A = oracle.fused_gemv_q4k(W, gate, up=up)
    check(q.qgemv_q4k_fused(dev(W), dev(gate), up=dev(up)).cpu().numpy(), Y, A, what="silu tails")
    x = synth.gen_x(1, K, 16) * 3.0e4
    g = synth.gen_x(1, K, 17)[0]
    Y, A = oracle.fused_gemv_q4k(W, x, norm_weight=g, eps=1e-6)
    check(q.qgemv_q4k_fused(dev(W), dev(x), norm_weight=dev(g), eps=1e-6).cpu().numpy(), Y, A, what="norm scale")


@pytest.mark.parametrize("N", [96, 9728])   # few tiles: two warps per column; 304 tiles: one warp per column
@pytest.mark.parametrize("scale", [2.0 ** 50, 2.0 ** -40])
def test_prologue_output_outside_direct_range(q, N, scale):
    """The prologue's output (x * g before 1/rms, silu(gate) * up) far
    outside [2^-24, 2^39): the staged column is rescaled by a power of two
    and its sums scaled back, in both fused kernels."""
    K = 2048
    W = synth.gen_q4k(N, K, 5000 + N)
    x = synth.gen_x(1, K, 18) * scale
    g = synth.gen_x(1, K, 19)[0]
    Y, A = oracle.fused_gemv_q4k(W, x, norm_weight=g, eps=0.0)
    y = q.qgemv_q4k_fused(dev(W), dev(x), norm_weight=dev(g), eps=0.0)
    check(y.cpu().numpy(), Y, A, what=f"rmsnorm N={N} x*{scale:g}")
    gate = synth.gen_x(1, K, 20)
    up = synth.gen_x(1, K, 21) * scale
    Y, A = oracle.fused_gemv_q4k(W, gate, up=up)
    y = q.qgemv_q4k_fused(dev(W), dev(gate), up=dev(up))
    check(y.cpu().numpy(), Y, A, what=f"swiglu N={N} up*{scale:g}")
    assert q.qg_device_status() == q.QG_OK


@pytest.mark.parametrize("flags", [0, 1])
def test_group_rmsnorm_qkv(q, flags):
    """q/k/v of one TinyLlama-shaped layer (2048 -> 2048, 256, 256) with the
    attention RMSNorm as one grouped launch."""
    K = 2048
    Ws = [synth.gen_q4k(n, K, 5000 + n) for n in (2048, 256, 256)]
    x = synth.gen_x(1, K, 18)
    g = synth.gen_x(1, K, 19)[0]
    outs = q.qgemv_q4k_fused_group([dev(w) for w in Ws], dev(x), norm_weight=dev(g), eps=1e-5, flags=flags)
    for W, y in zip(Ws, outs):
        Y, A = oracle.fused_gemv_q4k(W, x, norm_weight=g, eps=1e-5)
        check(y.cpu().numpy(), Y, A, what="qkv group")


def test_group_residual_per_matrix(q):
    K = 768
    Ws = [synth.gen_q4k(n, K, 6000 + n) for n in (40, 65)]
    x = synth.gen_x(2, K, 20)
    Rs = [synth.gen_x(2, n, 21 + n) for n in (40, 65)]
    outs = q.qgemv_q4k_fused_group([dev(w) for w in Ws], dev(x), residuals=(dev(Rs[0]), None))
    Y0, A0 = oracle.fused_gemv_q4k(Ws[0], x, residual=Rs[0])
    Y1, A1 = oracle.fused_gemv_q4k(Ws[1], x)
    check(outs[0].cpu().numpy(), Y0, A0, res=True, what="group residual 0")
    check(outs[1].cpu().numpy(), Y1, A1, what="group no residual 1")


def test_decode_step_chain(q):
    """Two layers of a small decode step, every GEMV fused and reading the
    previous GEMV's output on the device: q/k/v (attention RMSNorm) -> o
    (x = q, standing in for attention; residual in place) -> gate/up (FFN
    RMSNorm) -> down (SwiGLU, residual in place) -> output (final RMSNorm).
    The chain of programmatic dependent launches (no host synchronisation in
    between) equals, bit for bit, the same chain with the host waiting after
    every launch; and every stage, given the oracle's own chain of inputs
    (the fp32 of the oracle's previous outputs), matches the oracle."""
    D, F, KV, V = 512, 1024, 128, 600
    rng = np.random.default_rng(77)
    x0 = synth.gen_x(1, D, 30)
    layers = []
    for layer in range(2):
        Wq, Wk, Wv, Wo = (synth.gen_q4k(n, D, 7000 + 10 * layer + i) for i, n in enumerate((D, KV, KV, D)))
        Wg, Wu = (synth.gen_q4k(F, D, 7100 + 10 * layer + i) for i in range(2))
        Wd = synth.gen_q4k(D, F, 7200 + layer)
        ga, gf = (rng.standard_normal(D).astype(np.float32) for _ in range(2))
        layers.append((Wq, Wk, Wv, Wo, Wg, Wu, Wd, ga, gf))
    Wout = synth.gen_q4k(V, D, 7300)
    gn = rng.standard_normal(D).astype(np.float32)

    def gpu_chain(fl, wait):
        x = dev(x0)
        outs = []
        for Wq, Wk, Wv, Wo, Wg, Wu, Wd, ga, gf in layers:
            qv, kv, vv = q.qgemv_q4k_fused_group([dev(Wq), dev(Wk), dev(Wv)], x, norm_weight=dev(ga), eps=1e-5,
                                                 flags=fl)
            wait()
            q.qgemv_q4k_fused(dev(Wo), qv, out=x, residual=x, flags=fl)
            wait()
            x_mid = x.clone()
            gt, upv = q.qgemv_q4k_fused_group([dev(Wg), dev(Wu)], x, norm_weight=dev(gf), eps=1e-5, flags=fl)
            wait()
            q.qgemv_q4k_fused(dev(Wd), gt, out=x, up=upv, residual=x, flags=fl)
            wait()
            outs += [qv, kv, vv, x_mid, gt, upv, x.clone()]
        outs.append(q.qgemv_q4k_fused(dev(Wout), x, norm_weight=dev(gn), eps=1e-5, flags=fl))
        torch.cuda.synchronize()
        return outs

    chained = gpu_chain(q.QG_PREFETCH_WEIGHTS, lambda: None)
    stepped = gpu_chain(0, torch.cuda.synchronize)
    for a, b in zip(chained, stepped):
        assert torch.equal(a, b)
    assert q.qg_device_status() == 0

    # every stage on the oracle's chain of inputs
    def f32(Y):
        return np.asarray(Y, dtype=np.float32)

    x = x0
    for layer, (Wq, Wk, Wv, Wo, Wg, Wu, Wd, ga, gf) in enumerate(layers):
        outs = q.qgemv_q4k_fused_group([dev(Wq), dev(Wk), dev(Wv)], dev(x), norm_weight=dev(ga), eps=1e-5)
        refs = [oracle.fused_gemv_q4k(W, x, norm_weight=ga, eps=1e-5) for W in (Wq, Wk, Wv)]
        for o, (Y, A) in zip(outs, refs):
            check(o.cpu().numpy(), Y, A, what=f"{layer} qkv")
        qv = f32(refs[0][0])
        Y, A = oracle.fused_gemv_q4k(Wo, qv, residual=x)
        check(q.qgemv_q4k_fused(dev(Wo), dev(qv), residual=dev(x)).cpu().numpy(), Y, A, res=True, what=f"{layer} o")
        x = f32(Y)
        outs = q.qgemv_q4k_fused_group([dev(Wg), dev(Wu)], dev(x), norm_weight=dev(gf), eps=1e-5)
        refs = [oracle.fused_gemv_q4k(W, x, norm_weight=gf, eps=1e-5) for W in (Wg, Wu)]
        for o, (Y, A) in zip(outs, refs):
            check(o.cpu().numpy(), Y, A, what=f"{layer} gate/up")
        gt, upv = f32(refs[0][0]), f32(refs[1][0])
        Y, A = oracle.fused_gemv_q4k(Wd, gt, up=upv, residual=x)
        check(q.qgemv_q4k_fused(dev(Wd), dev(gt), up=dev(upv), residual=dev(x)).cpu().numpy(), Y, A, res=True,
              what=f"{layer} down")
        x = f32(Y)
    Y, A = oracle.fused_gemv_q4k(Wout, x, norm_weight=gn, eps=1e-5)
    check(q.qgemv_q4k_fused(dev(Wout), dev(x), norm_weight=dev(gn), eps=1e-5).cpu().numpy(), Y, A, what="output")
    assert q.qg_device_status() == 0
