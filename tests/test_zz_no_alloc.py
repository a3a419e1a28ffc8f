"""qgemv_q4k_pass_noalloc: the decode pass with its stage counts in the
library's fixed scratch array instead of caller memory.

Collected last on purpose (file name): it must pass alone in a fresh process
and after every other test, whatever state the shared scratch was left in.
"""
import numpy as np
import pytest

from block_quantised_weight_gb300 import build, qgemv, synth

TAU_FMA = 1e-5  # |y - y_ref| <= 1e-5 * sum|w*x|, as for every fp32 FMA-path test


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qgemv.load()


def test_noalloc_rejects_more_stages_than_scratch(lib):
    """Host-side checks only: nothing reaches the GPU."""
    n = qgemv.QG_NOALLOC_SCRATCH_WORDS + 1
    arr = (qgemv.QgStage * n)()
    assert lib.qgemv_q4k_pass_noalloc(arr, n, 1, None) == qgemv.QG_ESCRATCH
    assert "scratch" in qgemv.strerror(qgemv.QG_ESCRATCH)
    assert lib.qgemv_q4k_pass_noalloc(None, 1, 1, None) == qgemv.QG_EINVAL
    assert lib.qgemv_q4k_pass_noalloc(arr, 0, 1, None) == qgemv.QG_EINVAL
    assert lib.qgemv_q4k_pass_noalloc(arr, 1, 5, None) == qgemv.QG_EINVAL


def _chain(torch, Ws, M, x0):
    """Stages [A,B] <- x0, [C] <- yA, [D] <- yC, [E,F] <- yD with fresh outputs."""
    A, B, C, D, E, F = Ws
    ys = [torch.full((M, n), float("nan"), device="cuda") for n in (512, 256, 768, 256, 100, 64)]
    yA, yB, yC, yD, yE, yF = ys
    return [([A, B], [yA, yB], x0), ([C], [yC], yA), ([D], [yD], yC), ([E, F], [yE, yF], yD)]


@pytest.mark.gpu
def test_noalloc_matches_pass_on_two_calls_in_a_row(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(77)
    shapes = [(512, 512), (256, 512), (768, 512), (256, 768), (100, 256), (64, 256)]

    def weights():
        return [torch.from_numpy(synth.gen_q4k(n, k, rng)).cuda() for n, k in shapes]

    cases = []
    for M, seed in ((1, 3), (2, 4)):      # two different passes, issued back to back
        Ws = weights()
        x0 = torch.from_numpy(synth.gen_x(M, 512, seed)).cuda()
        cases.append((M, Ws, _chain(torch, Ws, M, x0), _chain(torch, Ws, M, x0)))

    for M, _, mine, _ in cases:           # the two calls, no synchronisation between them
        qgemv.qgemv_q4k_pass_noalloc(mine, M=M)
    sync = torch.zeros(8, dtype=torch.int32, device="cuda")
    for M, _, _, ref in cases:
        qgemv.qgemv_q4k_pass(ref, sync, M=M)
    torch.cuda.synchronize()

    for M, Ws, mine, ref in cases:
        for (_, ys, _), (Wr, yr, Xr) in zip(mine, ref):
            for W, y, y_ref in zip(Wr, ys, yr):
                K = Xr.shape[-1]
                scale = qgemv.qdequant_q4k(W, K).abs() @ Xr.reshape(M, K).abs().T   # sum|w*x|, [N, M]
                err = (y - y_ref).abs().T
                assert torch.isfinite(y).all()
                assert bool((err <= TAU_FMA * scale).all()), f"M={M}: worst {float(err.max()):.3e}"
    assert qgemv.qg_device_status() == qgemv.QG_OK
