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
    previous GEMV's output on the device (programmatic dependent launches,
    no host synchronisation in between): q/k/v (attention RMSNorm) -> o
    (x = q, standing in for attention; residual in place) -> gate/up (FFN
    RMSNorm) -> down (SwiGLU, residual in place) -> output (final RMSNorm).
    Device-side snapshots record what each stage read and wrote; every stage
    is then checked against the oracle on the inputs the GPU gave it."""
    D, F, KV, V = 512, 1024, 128, 600
    rng = np.random.default_rng(77)
    x = dev(synth.gen_x(1, D, 30))
    fl = q.QG_PREFETCH_WEIGHTS
    stages = []  # (name, [W], oracle kwargs with device snapshots, [output snapshots], residual?)
    for layer in range(2):
        Wq, Wk, Wv, Wo = (synth.gen_q4k(n, D, 7000 + 10 * layer + i) for i, n in enumerate((D, KV, KV, D)))
        Wg, Wu = (synth.gen_q4k(F, D, 7100 + 10 * layer + i) for i in range(2))
        Wd = synth.gen_q4k(D, F, 7200 + layer)
        ga, gf = (rng.standard_normal(D).astype(np.float32) for _ in range(2))
        x_in = x.clone()
        qv, kv, vv = q.qgemv_q4k_fused_group([dev(Wq), dev(Wk), dev(Wv)], x, norm_weight=dev(ga), eps=1e-5,
                                             flags=fl)
        stages.append((f"{layer} qkv", [Wq, Wk, Wv], dict(X=x_in, norm_weight=ga, eps=1e-5),
                       [qv.clone(), kv.clone(), vv.clone()], False))
        x_before = x.clone()
        q.qgemv_q4k_fused(dev(Wo), qv, out=x, residual=x, flags=fl)
        stages.append((f"{layer} o", [Wo], dict(X=qv.clone(), residual=x_before), [x.clone()], True))
        x_mid = x.clone()
        gt, upv = q.qgemv_q4k_fused_group([dev(Wg), dev(Wu)], x, norm_weight=dev(gf), eps=1e-5, flags=fl)
        stages.append((f"{layer} gate/up", [Wg, Wu], dict(X=x_mid, norm_weight=gf, eps=1e-5),
                       [gt.clone(), upv.clone()], False))
        q.qgemv_q4k_fused(dev(Wd), gt, out=x, up=upv, residual=x, flags=fl)
        stages.append((f"{layer} down", [Wd], dict(X=gt.clone(), up=upv.clone(), residual=x_mid.clone()),
                       [x.clone()], True))
    Wout = synth.gen_q4k(V, D, 7300)
    gn = rng.standard_normal(D).astype(np.float32)
    x_fin = x.clone()
    logits = q.qgemv_q4k_fused(dev(Wout), x, norm_weight=dev(gn), eps=1e-5, flags=fl)
    stages.append(("output", [Wout], dict(X=x_fin, norm_weight=gn, eps=1e-5), [logits], False))
    assert q.qg_device_status() == 0
    for name, Ws, kw, outs, res in stages:
        kw = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
        X = kw.pop("X")
        for W, o in zip(Ws, outs):
            Y, A = oracle.fused_gemv_q4k(W, X, **kw)
            check(o.cpu().numpy(), Y, A, res=res, what=name)
