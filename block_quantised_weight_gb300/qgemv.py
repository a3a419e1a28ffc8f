"""ctypes binding of libqgemv.so: argument marshalling only.

Each function takes torch CUDA tensors, checks dtype/shape/contiguity, and
calls the C entry point of the same name on the current torch stream (or the
stream given).  Every step of the computation runs in the library's CUDA
kernels; there is no CPU fallback: if the library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

QG_OK = 0
QG_EINVAL = -1
QG_EALIGN = -2
QG_ECUDA = -3
QG_ETIMEOUT = -4
QG_EBOUNDS = -5
QG_EALIAS = -6
QG_ESCRATCH = -7
QG_MAX_M = 32
QG_MAX_GROUP = 4
QG_MAX_PASS_STAGES = 96
QG_NOALLOC_SCRATCH_WORDS = 96


class QgStage(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p * 4), ("Y", ctypes.c_void_p * 4), ("N", ctypes.c_int64 * 4),
                ("count", ctypes.c_int), ("X", ctypes.c_void_p), ("K", ctypes.c_int64)]

class QgFuse(ctypes.Structure):
    _fields_ = [("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float), ("up", ctypes.c_void_p),
                ("residual", ctypes.c_void_p * 4)]

QG_PREFETCH_WEIGHTS = 1
QG_CB = {"iq4nl": 1, "iq4xs": 2, "iq3s": 3, "iq2xxs": 4}
CB_UNIT_BYTES = {"iq4nl": 144, "iq4xs": 136, "iq3s": 110, "iq2xxs": 66}

EXPORTS = ("qgemv_q4k", "qgemv_q4k_ex", "qgemv_q4k_group", "qgemv_q4k_fused", "qgemv_q4k_fused_group", "qgemv_q4k_pass", "qgemv_q4k_pass_noalloc", "qgemv_iq3", "qgemv_iq3_ex", "qgemv_iq3_group", "qgemv_iq3xxs", "qgemv_iq3xxs_ex", "qdequant_iq3xxs", "qgemv_codebook", "qdequant_codebook", "qgemm_q4k_batched", "qgemm_iq3_batched", "qdequant_q4k", "qdequant_iq3",
           "qg_device_status", "qg_test_bounded_wait", "qg_test_chain_step", "qg_strerror", "qg_last_cuda_error")


class QGError(RuntimeError):
    def __init__(self, fn: str, code: int, cuda_error: int = 0):
        self.code = code
        self.cuda_error = cuda_error
        extra = f"; cudaError {cuda_error}" if code == QG_ECUDA and cuda_error else ""
        super().__init__(f"{fn} failed: {code} ({strerror(code)}{extra})")


def library_path() -> str:
    return _build.LIB


def load():
    """Load libqgemv.so (built in-tree by build.build()); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libqgemv.so is not built ({path}); run block_quantised_weight_gb300.build.build()")
        lib = ctypes.CDLL(path)
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        sigs = {
            "qgemv_q4k": [vp, vp, vp, ci, i64, i64, vp],
            "qgemv_q4k_ex": [vp, vp, vp, ci, i64, i64, ctypes.c_uint, vp],
            "qgemv_iq3": [vp, vp, vp, vp, ci, i64, i64, vp],
            "qgemv_iq3_ex": [vp, vp, vp, vp, ci, i64, i64, ctypes.c_uint, vp],
            "qgemv_iq3xxs": [vp, vp, vp, vp, ci, i64, i64, vp],
            "qgemv_iq3xxs_ex": [vp, vp, vp, vp, ci, i64, i64, ctypes.c_uint, vp],
            "qdequant_iq3xxs": [vp, vp, vp, i64, i64, vp],
            "qgemv_codebook": [ci, vp, vp, vp, vp, ci, i64, i64, vp],
            "qdequant_codebook": [ci, vp, vp, vp, i64, i64, vp],
            "qgemv_q4k_group": [vp, vp, vp, ci, vp, ci, i64, ctypes.c_uint, vp],
            "qgemv_iq3_group": [vp, vp, vp, ci, vp, vp, ci, i64, ctypes.c_uint, vp],
            "qgemv_q4k_fused": [vp, vp, vp, ci, i64, i64, vp, ctypes.c_uint, vp],
            "qgemv_q4k_fused_group": [vp, vp, vp, ci, vp, ci, i64, vp, ctypes.c_uint, vp],
            "qgemv_q4k_pass": [vp, ci, ci, vp, vp],
            "qgemv_q4k_pass_noalloc": [vp, ci, ci, vp],
            "qgemm_q4k_batched": [vp, vp, vp, ci, i64, i64, vp],
            "qgemm_iq3_batched": [vp, vp, vp, vp, ci, i64, i64, vp],
            "qdequant_q4k": [vp, vp, i64, i64, vp],
            "qdequant_iq3": [vp, vp, vp, i64, i64, vp],
            "qg_device_status": [vp],
            "qg_test_bounded_wait": [vp],
            "qg_test_chain_step": [vp, vp, i64, ci, ctypes.c_uint, vp],
            "qg_strerror": [ci],
            "qg_last_cuda_error": [],
        }
        for name, args in sigs.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_char_p if name == "qg_strerror" else ctypes.c_int
        _lib = lib
        return lib


def strerror(code: int) -> str:
    try:
        return load().qg_strerror(int(code)).decode()
    except Exception:  # library not loadable: still give a message
        return "unknown"


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _check(fn, rc):
    if rc != QG_OK:
        # the CUDA error behind a QG_ECUDA, recorded for this host thread
        raise QGError(fn, rc, int(load().qg_last_cuda_error()) if rc == QG_ECUDA else 0)


def _req(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _xy(W, X, out, block_bytes):
    import torch
    _req(W, torch.uint8, "W")
    _req(X, torch.float32, "X")
    if X.dim() == 1:
        X = X.view(1, -1)
    M, K = X.shape
    if K % 256:
        raise ValueError("K must be a multiple of 256")
    row = K // 256 * block_bytes
    if W.numel() % row:
        raise ValueError("W is not a whole number of rows for this K")
    N = W.numel() // row
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=X.device)
    else:
        _req(out, torch.float32, "out")
        if out.numel() != M * N:
            raise ValueError("out has the wrong size")
    return X, out, M, N, K


def qgemv_q4k(W, X, out=None, stream=None, flags=0):
    """Y[M, N] = X[M, K] @ dequant(W)^T for a Q4_K matrix W (uint8, N*K/256*144 bytes).

    flags=QG_PREFETCH_WEIGHTS calls qgemv_q4k_ex (programmatic dependent launch)."""
    X, out, M, N, K = _xy(W, X, out, 144)
    if flags:
        rc = load().qgemv_q4k_ex(W.data_ptr(), X.data_ptr(), out.data_ptr(), M, N, K, flags, _stream(stream))
        _check("qgemv_q4k_ex", rc)
    else:
        _check("qgemv_q4k", load().qgemv_q4k(W.data_ptr(), X.data_ptr(), out.data_ptr(), M, N, K, _stream(stream)))
    return out


def qgemv_iq3(W, grid, X, out=None, stream=None, flags=0):
    """Y[M, N] = X @ dequant(W)^T for an IQ3 matrix W with codebook grid (uint8 [256, 4], doubled units)."""
    import torch
    _req(grid, torch.uint8, "grid")
    if grid.numel() != 1024:
        raise ValueError("grid must hold 256 x 4 bytes")
    X, out, M, N, K = _xy(W, X, out, 98)
    rc = load().qgemv_iq3_ex(W.data_ptr(), grid.data_ptr(), X.data_ptr(), out.data_ptr(), M, N, K, flags,
                             _stream(stream))
    _check("qgemv_iq3_ex" if flags else "qgemv_iq3", rc)
    return out


def qgemv_iq3xxs(W, grid, X, out=None, stream=None, flags=0):
    """Y = X @ dequant(W)^T for an IQ3_XXS matrix (page 3 byte order, raw grid entries)."""
    import torch
    _req(grid, torch.uint8, "grid")
    if grid.numel() != 1024:
        raise ValueError("grid must hold 256 x 4 bytes")
    X, out, M, N, K = _xy(W, X, out, 98)
    rc = load().qgemv_iq3xxs_ex(W.data_ptr(), grid.data_ptr(), X.data_ptr(), out.data_ptr(), M, N, K, flags,
                                _stream(stream))
    _check("qgemv_iq3xxs_ex", rc)
    return out


def qgemv_codebook(fmt, W, codebook, X, out=None, stream=None):
    """Y = X @ dequant(W)^T for page 3's codebook formats ("iq4nl", "iq4xs",
    "iq3s", "iq2xxs"); codebook: int8 [16] or uint8 [512, 4] / [256, 8]."""
    _req(codebook, codebook.dtype, "codebook")
    X, out, M, N, K = _xy(W, X, out, CB_UNIT_BYTES[fmt])
    rc = load().qgemv_codebook(QG_CB[fmt], W.data_ptr(), codebook.data_ptr(), X.data_ptr(), out.data_ptr(), M, N, K,
                               _stream(stream))
    _check("qgemv_codebook", rc)
    return out


def qdequant_codebook(fmt, W, codebook, K, out=None, stream=None):
    """Test-only: fp32 [N, K] dequantisation of a codebook-format matrix."""
    import torch
    _req(W, torch.uint8, "W")
    N = W.numel() // (K // 256 * CB_UNIT_BYTES[fmt])
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=W.device)
    _check("qdequant_codebook", load().qdequant_codebook(QG_CB[fmt], W.data_ptr(), codebook.data_ptr(),
                                                         out.data_ptr(), N, K, _stream(stream)))
    return out


def group_arrays(Ws, Ys, Ns):
    """Host arrays (kept alive by the caller) of device pointers and row counts."""
    n = len(Ws)
    Wa = (ctypes.c_void_p * n)(*[w.data_ptr() for w in Ws])
    Ya = (ctypes.c_void_p * n)(*[y.data_ptr() for y in Ys])
    Na = (ctypes.c_int64 * n)(*Ns)
    return Wa, Ya, Na


def qgemv_q4k_group(Ws, X, outs=None, stream=None, flags=0):
    """[X @ dequant(W_i)^T for W_i in Ws] (all W_i share K): one launch per token
    group of up to 4 on the FMA path; from 5 tokens one tensor-core launch per
    matrix and group of up to 10."""
    import torch
    Xv = X.view(1, -1) if X.dim() == 1 else X
    M, K = Xv.shape
    Ns = []
    for W in Ws:
        _req(W, torch.uint8, "W")
        Ns.append(W.numel() // (K // 256 * 144))
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.float32, device=X.device) for n in Ns]
    _req(Xv, torch.float32, "X")
    Wa, Ya, Na = group_arrays(Ws, outs, Ns)
    rc = load().qgemv_q4k_group(Wa, Ya, Na, len(Ws), Xv.data_ptr(), M, K, flags, _stream(stream))
    _check("qgemv_q4k_group", rc)
    return outs


def qgemv_iq3_group(Ws, grid, X, outs=None, stream=None, flags=0):
    """IQ3 counterpart of qgemv_q4k_group (one grid)."""
    import torch
    Xv = X.view(1, -1) if X.dim() == 1 else X
    M, K = Xv.shape
    Ns = []
    for W in Ws:
        _req(W, torch.uint8, "W")
        Ns.append(W.numel() // (K // 256 * 98))
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.float32, device=X.device) for n in Ns]
    _req(Xv, torch.float32, "X")
    _req(grid, torch.uint8, "grid")
    Wa, Ya, Na = group_arrays(Ws, outs, Ns)
    rc = load().qgemv_iq3_group(Wa, Ya, Na, len(Ws), grid.data_ptr(), Xv.data_ptr(), M, K, flags, _stream(stream))
    _check("qgemv_iq3_group", rc)
    return outs


def fuse_struct(norm_weight=None, eps=0.0, up=None, residuals=()):
    """qg_fuse from torch CUDA tensors (None disables an operand)."""
    import torch
    f = QgFuse()
    if norm_weight is not None:
        _req(norm_weight, torch.float32, "norm_weight")
        f.norm_weight = norm_weight.data_ptr()
    f.norm_eps = float(eps)
    if up is not None:
        _req(up, torch.float32, "up")
        f.up = up.data_ptr()
    for i, r in enumerate(residuals):
        if r is not None:
            _req(r, torch.float32, "residual")
            f.residual[i] = r.data_ptr()
    return f


def qgemv_q4k_fused(W, X, out=None, norm_weight=None, eps=0.0, up=None, residual=None, stream=None, flags=0):
    """Y = h @ dequant(W)^T (+ residual) with h = X, rmsnorm(X; norm_weight, eps)
    or silu(X) * up (qgemv_q4k_fused).  residual may be `out` itself."""
    X, out, M, N, K = _xy(W, X, out, 144)
    f = fuse_struct(norm_weight, eps, up, (residual,))
    rc = load().qgemv_q4k_fused(W.data_ptr(), X.data_ptr(), out.data_ptr(), M, N, K, ctypes.byref(f), flags,
                                _stream(stream))
    _check("qgemv_q4k_fused", rc)
    return out


def qgemv_q4k_fused_group(Ws, X, outs=None, norm_weight=None, eps=0.0, up=None, residuals=(), stream=None,
                          flags=0):
    """qgemv_q4k_group with a shared prologue and per-matrix residuals."""
    import torch
    Xv = X.view(1, -1) if X.dim() == 1 else X
    M, K = Xv.shape
    Ns = []
    for W in Ws:
        _req(W, torch.uint8, "W")
        Ns.append(W.numel() // (K // 256 * 144))
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.float32, device=X.device) for n in Ns]
    _req(Xv, torch.float32, "X")
    Wa, Ya, Na = group_arrays(Ws, outs, Ns)
    f = fuse_struct(norm_weight, eps, up, residuals)
    rc = load().qgemv_q4k_fused_group(Wa, Ya, Na, len(Ws), Xv.data_ptr(), M, K, ctypes.byref(f), flags,
                                      _stream(stream))
    _check("qgemv_q4k_fused_group", rc)
    return outs


def pass_stages(stages):
    """ctypes array of qg_stage from [(Ws, Ys, X)] (torch CUDA tensors)."""
    arr = (QgStage * len(stages))()
    for i, (Ws, Ys, X) in enumerate(stages):
        Xv = X.view(1, -1) if X.dim() == 1 else X
        K = Xv.shape[1]
        st = arr[i]
        st.count = len(Ws)
        for j, (W, Y) in enumerate(zip(Ws, Ys)):
            st.W[j] = W.data_ptr()
            st.Y[j] = Y.data_ptr()
            st.N[j] = W.numel() // (K // 256 * 144)
        st.X = Xv.data_ptr()
        st.K = K
    return arr


def qgemv_q4k_pass(stages, sync, M=1, stream=None):
    """Run [(Ws, Ys, X)] stages as one persistent launch; sync: int32 CUDA tensor
    with at least len(stages) elements (zeroed by the call)."""
    import torch
    _req(sync, torch.int32, "sync")
    if sync.numel() < len(stages):
        raise ValueError("sync needs one word per stage")
    arr = pass_stages(stages)
    rc = load().qgemv_q4k_pass(arr, len(stages), M, sync.data_ptr(), _stream(stream))
    _check("qgemv_q4k_pass", rc)


def qgemv_q4k_pass_noalloc(stages, M=1, stream=None):
    """qgemv_q4k_pass with the stage counts in the library's fixed scratch:
    the call allocates nothing on the device.  Calls that overlap on the GPU
    race on that scratch."""
    arr = pass_stages(stages)
    rc = load().qgemv_q4k_pass_noalloc(arr, len(stages), M, _stream(stream))
    _check("qgemv_q4k_pass_noalloc", rc)


def qgemm_q4k_batched(W, X, out=None, stream=None):
    """Batched Q4_K GEMM: M < 16 as qgemv_q4k (fp32 FMA path up to 4 tokens, tensor
    cores with exact products from 5), M >= 16 on tcgen05 with bf16 weights."""
    X, out, M, N, K = _xy(W, X, out, 144)
    _check("qgemm_q4k_batched", load().qgemm_q4k_batched(W.data_ptr(), X.data_ptr(), out.data_ptr(), M, N, K,
                                                         _stream(stream)))
    return out


def qgemm_iq3_batched(W, grid, X, out=None, stream=None):
    """Batched IQ3 GEMM: with K/256 a multiple of 8, from 5 tokens on tcgen05 with the
    weights exact (x in three bf16 parts below 16 tokens, rounded to bf16 from
    16); otherwise the fp32 FMA path."""
    import torch
    _req(grid, torch.uint8, "grid")
    X, out, M, N, K = _xy(W, X, out, 98)
    _check("qgemm_iq3_batched", load().qgemm_iq3_batched(W.data_ptr(), grid.data_ptr(), X.data_ptr(),
                                                         out.data_ptr(), M, N, K, _stream(stream)))
    return out


def qdequant_q4k(W, K, out=None, stream=None):
    """Test-only: fp32 [N, K] dequantisation of a Q4_K matrix."""
    import torch
    _req(W, torch.uint8, "W")
    N = W.numel() // (K // 256 * 144)
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=W.device)
    _check("qdequant_q4k", load().qdequant_q4k(W.data_ptr(), out.data_ptr(), N, K, _stream(stream)))
    return out


def qdequant_iq3(W, grid, K, out=None, stream=None):
    """Test-only: fp32 [N, K] dequantisation of an IQ3 matrix."""
    import torch
    _req(W, torch.uint8, "W")
    _req(grid, torch.uint8, "grid")
    N = W.numel() // (K // 256 * 98)
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=W.device)
    _check("qdequant_iq3", load().qdequant_iq3(W.data_ptr(), grid.data_ptr(), out.data_ptr(), N, K,
                                               _stream(stream)))
    return out


def qdequant_iq3xxs(W, grid, K, out=None, stream=None):
    """Test-only: fp32 [N, K] dequantisation of an IQ3_XXS matrix."""
    import torch
    _req(W, torch.uint8, "W")
    _req(grid, torch.uint8, "grid")
    N = W.numel() // (K // 256 * 98)
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=W.device)
    _check("qdequant_iq3xxs", load().qdequant_iq3xxs(W.data_ptr(), grid.data_ptr(), out.data_ptr(), N, K,
                                                     _stream(stream)))
    return out


def qg_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(load().qg_device_status(_stream(stream)))


def qg_test_bounded_wait(stream=None) -> int:
    return int(load().qg_test_bounded_wait(_stream(stream)))
