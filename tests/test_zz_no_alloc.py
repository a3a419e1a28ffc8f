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


def oracle_chain(host, x0):
    """The chain's stage inputs computed by the oracle alone: x0, then the fp32
    of the oracle's A, C and D outputs (what stages 2-4 read)."""
    import oracle
    A, B, C, D, E, F = host
    xs = [x0]
    for W in (A, C, D):
        Y, _ = oracle.gemv_q4k(W, xs[-1])
        xs.append(Y.astype(np.float32))
    return xs


@pytest.mark.gpu
def test_noalloc_matches_pass_on_two_calls_in_a_row(lib):
    """Two no-allocation passes issued back to back (different M, no
    synchronisation between them) give exactly what qgemv_q4k_pass gives: the
    same kernel, plan and grid, and no atomics in Y, so the outputs are equal
    bit for bit.  The same entry point, given the oracle's own stage inputs
    in place of the previous stages' outputs, matches the oracle within
    1e-5 * sum|w*x| on every output."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    rng = np.random.default_rng(77)
    shapes = [(512, 512), (256, 512), (768, 512), (256, 768), (100, 256), (64, 256)]

    cases = []
    for M, seed in ((1, 3), (2, 4)):      # two different passes, issued back to back
        host = [synth.gen_q4k(n, k, rng) for n, k in shapes]
        Ws = [torch.from_numpy(W).cuda() for W in host]
        x0 = torch.from_numpy(synth.gen_x(M, 512, seed)).cuda()
        cases.append((M, host, Ws, _chain(torch, Ws, M, x0), _chain(torch, Ws, M, x0)))

    for M, _, _, mine, _ in cases:        # the two calls, no synchronisation between them
        qgemv.qgemv_q4k_pass_noalloc(mine, M=M)
    sync = torch.zeros(8, dtype=torch.int32, device="cuda")
    for M, _, _, _, ref in cases:
        qgemv.qgemv_q4k_pass(ref, sync, M=M)
    torch.cuda.synchronize()
    for M, _, _, mine, ref in cases:
        for (_, ys, _), (_, yr, _) in zip(mine, ref):
            for y, y_ref in zip(ys, yr):
                assert torch.isfinite(y).all()
                assert torch.equal(y, y_ref), f"M={M}: the no-allocation pass differs from qgemv_q4k_pass"

    for M, host, Ws, mine, _ in cases:
        xs = oracle_chain(host, mine[0][2].cpu().numpy())
        A, B, C, D, E, F = Ws
        stages = [([A, B], [torch.empty((M, 512), device="cuda"), torch.empty((M, 256), device="cuda")]),
                  ([C], [torch.empty((M, 768), device="cuda")]),
                  ([D], [torch.empty((M, 256), device="cuda")]),
                  ([E, F], [torch.empty((M, 100), device="cuda"), torch.empty((M, 64), device="cuda")])]
        qgemv.qgemv_q4k_pass_noalloc([(w, y, torch.from_numpy(x).cuda()) for (w, y), x in zip(stages, xs)], M=M)
        torch.cuda.synchronize()
        hi = iter(host)
        for (_, ys), x in zip(stages, xs):
            for y in ys:
                Y, Ab = oracle.gemv_q4k(next(hi), x)
                err = np.abs(y.cpu().numpy().astype(np.float64) - Y)
                assert (err <= TAU_FMA * Ab).all(), f"M={M}: worst {float((err / Ab).max()):.3e} of sum|w*x|"
    assert qgemv.qg_device_status() == qgemv.QG_OK
