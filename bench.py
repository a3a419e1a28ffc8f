#!/usr/bin/env python3
"""Benchmark of the fused-dequantisation GEMV path (one JSON line on rank 0).

Headline workload: the TinyLlama-1.1B-shaped decode weight pass at M=1, Q4_K
throughout: 22 layers x (q, k, v, o, gate, up, down) + the output projection,
155 GEMVs, 581,861,376 weight bytes, seeded synthetic weights and x.  One
step = one pass.  value = effective weight GB/s (weight bytes / step time,
summed over ranks); tokens/s-equiv = passes per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload tinyllama|q4k_c0|iq3_c2|q4k_c3|q4k_c4a|q4k_c4b|iq3_c4a|iq3_c4b] [--M m]

The timed region replays a CUDA graph of the pass K times between CUDA
events on the launching stream; the graph also holds an event pair around
every launch, which gives the per-launch kernel durations used for the
roofline.  The pass reads 581 MB, more than the 126 MB L2, so every step
streams from HBM; single-matrix workloads rotate over enough copies to
exceed twice the L2.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective weight GB/s (% of HBM peak) for Q4_K/IQ3 GEMV at M=1; tokens/s-equiv"
Q4K_BYTES, IQ3_BYTES = 144, 98
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ workloads
def workload_spec(name: str, M: int):
    """[(fmt, K, N)] GEMVs of one step, a description, and the token count."""
    from block_quantised_weight_gb300 import synth
    if name == "tinyllama":
        mats = [("q4k", K, N) for (_l, _n, K, N) in synth.tinyllama_shapes()]
        return mats, "TinyLlama-1.1B-shaped Q4_K decode weight pass, M=1 (155 GEMVs, 581,861,376 weight bytes)", 1
    table = {
        "q4k_c0": ("q4k", 2048, 2048), "iq3_c2": ("iq3", 4096, 14336), "q4k_c3": ("q4k", 4096, 11008),
        "q4k_c4a": ("q4k", 8192, 28672), "q4k_c4b": ("q4k", 28672, 8192),
        "iq3_c4a": ("iq3", 8192, 28672), "iq3_c4b": ("iq3", 28672, 8192),
        # page 3's formats at the IQ3 config's shape (not headline configs)
        "iq3xxs_c2": ("iq3xxs", 4096, 14336), "iq4nl_c2": ("iq4nl", 4096, 14336),
        "iq4xs_c2": ("iq4xs", 4096, 14336), "iq3s_c2": ("iq3s", 4096, 14336),
        "iq2xxs_c2": ("iq2xxs", 4096, 14336),
    }
    fmt, K, N = table[name]
    return [(fmt, K, N)], f"{fmt.upper()} GEMV K={K} N={N} M={M}", M


def pass_groups(name, n, single):
    """Index groups launched together.  TinyLlama pass: per layer (q, k, v),
    (o), (gate, up), (down), then (output): 89 launches for 155 GEMVs."""
    if name != "tinyllama" or single:
        return [[i] for i in range(n)]
    groups = []
    for l in range(22):
        b = 7 * l
        groups += [[b, b + 1, b + 2], [b + 3], [b + 4, b + 5], [b + 6]]
    groups.append([154])
    return groups


UNIT_BYTES = {"q4k": Q4K_BYTES, "iq3": IQ3_BYTES, "iq3xxs": IQ3_BYTES, "iq4nl": 144, "iq4xs": 136, "iq3s": 110,
              "iq2xxs": 66}
CB_FORMATS = ("iq4nl", "iq4xs", "iq3s", "iq2xxs")


def weight_bytes(fmt, K, N):
    return N * (K // 256) * UNIT_BYTES[fmt]


def gen_mats(name, mats, M):
    """Host arrays per GEMV: (fmt, K, N, W, grid, x)."""
    import numpy as np
    from block_quantised_weight_gb300 import synth
    out = []
    if name == "tinyllama":
        for (_shape, rng), (fmt, K, N) in zip(synth.tinyllama_seeds(1), mats):
            W = synth.gen_q4k(N, K, rng)
            x = synth.gen_x(M, K, rng)
            out.append((fmt, K, N, W, None, x))
        return out
    fmt, K, N = mats[0]
    seed = {"q4k_c0": 0, "iq3_c2": 2, "q4k_c3": 3}.get(name, 4)
    rng = np.random.default_rng(seed)
    if fmt == "q4k":
        W, grid = synth.gen_q4k(N, K, rng), None
    elif fmt in CB_FORMATS:
        W, grid = synth.gen_cb(fmt, N, K, rng)
    else:  # IQ3 fields; the page-3 order is the same bytes with d moved first
        W, grid = synth.gen_iq3(N, K, rng)
        if fmt == "iq3xxs":
            b = W.reshape(N, K // 256, 98)
            W = np.concatenate([b[:, :, 96:98], b[:, :, 0:96]], axis=2).reshape(N, -1)
    x = synth.gen_x(M, K, rng)
    out.append((fmt, K, N, W, grid, x))
    return out


# ------------------------------------------------------------------ helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l.split(",") for l in self.lines if l.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def cudart():
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


# Sources each kernel is built from (the library's translation unit for it
# and everything that unit includes).
_COMMON = ["common.cuh", "gemv_kernel.cuh", "launch.h", "tensor_map.h", "launch_common.cuh",
           "../../include/qgemv.h"]
KERNEL_SOURCES = {
    "q4k": _COMMON + ["launch_q4k.cuh", "gemv_q4k.cu"],
    "iq3": _COMMON + ["launch_iq3.cuh", "gemv_iq3.cu"],
    "tc": ["common.cuh", "gemv_kernel.cuh", "launch.h", "tensor_map.h", "../../include/qgemv.h", "gemm_tc.cu",
           "launch_q4k.cuh", "launch_iq3.cuh"],
    "cb": _COMMON + ["gemv_cb.cu"],
}


def kernel_source_hash(files=None):
    """Hash of the given kernel sources (paths relative to csrc/), or of every
    source in csrc/."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantised_weight_gb300", "csrc")
    if files is None:
        files = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, M):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary,
    only if that kernel's sources are unchanged since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
        e = d.get(f"{workload}:M{M}")
        if e and e.get("kernel_source_hash") == kernel_source_hash(KERNEL_SOURCES[e["sources"]]):
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ ranks
def max_over_ranks(vals, world, device):
    """Every rank's timings -> the slowest rank's, on every rank.  Replicas
    share no data; this and a barrier are the only collectives."""
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_throughput(world, bytes_per_step, steps, ms):
    """Whole-job GB/s: every replica streams bytes_per_step per step, all in
    the slowest rank's time."""
    return world * bytes_per_step * steps / (ms * 1e-3) / 1e9


def kernel_launches(lib, fn, a, M):
    """Kernels of ours that one C-ABI call launches: the FMA paths split M
    into token groups (Q4_K, IQ3 and the IQ4 codebook formats 4, the other
    codebook formats 8), each a launch; the batched tcgen05 path (M >= 16)
    and the persistent pass are one launch; Q4_K (without prologue or
    residual) and IQ3 (rows a multiple of 16 bytes, every workload here)
    from 5 tokens below 16 one tcgen05 launch per matrix and group of at most
    10 tokens."""
    if fn in (lib.qgemm_q4k_batched, lib.qgemm_iq3_batched) and M >= 16:
        return 1
    if fn in (lib.qgemv_q4k_ex, lib.qgemm_q4k_batched, lib.qgemv_iq3_ex, lib.qgemm_iq3_batched) and M >= 5:
        return (M + 9) // 10
    if fn in (lib.qgemv_q4k_group, lib.qgemv_iq3_group) and M >= 5:
        return a[3] * ((M + 9) // 10)
    if fn in (lib.qgemv_q4k_ex, lib.qgemv_q4k_group, lib.qgemv_q4k_fused, lib.qgemv_q4k_fused_group,
              lib.qgemm_q4k_batched):
        return (M + 3) // 4
    if fn in (lib.qgemv_iq3_ex, lib.qgemv_iq3_group, lib.qgemv_iq3xxs_ex, lib.qgemm_iq3_batched):
        return (M + 3) // 4  # rows a multiple of 16 bytes (every workload here)
    if fn == lib.qgemv_codebook:
        return (M + 3) // 4 if a[0] in (1, 2) else (M + 7) // 8
    return 1


# ------------------------------------------------------------------ our arm
def fused_step_launches(lib, qgemv, host, dev, keep):
    """The TinyLlama-shaped decode step with its data flow on the device, every
    GEMV fused (page 2 "Candle", Block::forward; page 1 model_forward): per
    layer q/k/v = rmsnorm(x) W^T (one grouped launch), x += q Wo^T (q stands
    in for the attention output, which is outside this library), gate/up =
    rmsnorm(x) W^T (grouped), x += (silu(gate) * up) Wd^T; then logits =
    rmsnorm(x) Wout^T.  89 launches, the weights of the plain pass; the norm
    weights are seeded 1 + 0.1 N(0, 1).  Returns (launches, x, logits, x0)."""
    import numpy as np
    import torch
    rng = np.random.default_rng(12345)
    D = host[0][1]
    mats = [torch.from_numpy(h[3]).to(dev) for h in host]
    keep.extend(mats)
    x0 = host[0][5].reshape(-1).astype(np.float32)
    x = torch.from_numpy(x0.copy()).to(dev)
    qkv = [torch.empty(h[2], dtype=torch.float32, device=dev) for h in host[0:3]]
    gu = [torch.empty(h[2], dtype=torch.float32, device=dev) for h in host[4:6]]
    logits = torch.empty(host[154][2], dtype=torch.float32, device=dev)
    keep.extend([x, logits, *qkv, *gu])
    fl = qgemv.QG_PREFETCH_WEIGHTS
    lst = []

    def fz(norm=None, up=None, res=None):
        f = qgemv.fuse_struct(norm, 1e-5, up, (res,))
        keep.append(f)
        return ctypes.byref(f)

    def norm_w():
        g = torch.from_numpy((1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)).to(dev)
        keep.append(g)
        return g

    for l in range(22):
        b = 7 * l
        ws = [mats[b + i] for i in range(7)]
        Ns = [host[b + i][2] for i in range(7)]
        Wa = (ctypes.c_void_p * 3)(*[w.data_ptr() for w in ws[0:3]])
        Ya = (ctypes.c_void_p * 3)(*[t.data_ptr() for t in qkv])
        Na = (ctypes.c_int64 * 3)(*Ns[0:3])
        Wb = (ctypes.c_void_p * 2)(*[w.data_ptr() for w in ws[4:6]])
        Yb = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in gu])
        Nb = (ctypes.c_int64 * 2)(*Ns[4:6])
        keep.append((Wa, Ya, Na, Wb, Yb, Nb))
        F = host[b + 4][2]
        wq = sum(weight_bytes("q4k", D, n) for n in Ns[0:3])
        lst.append((lib.qgemv_q4k_fused_group, (Wa, Ya, Na, 3, x.data_ptr(), 1, D, fz(norm=norm_w()), fl), wq,
                    wq + 8 * D + 4 * sum(Ns[0:3]), "fused qkv+rmsnorm"))
        wo = weight_bytes("q4k", D, D)
        lst.append((lib.qgemv_q4k_fused, (ws[3].data_ptr(), qkv[0].data_ptr(), x.data_ptr(), 1, D, D,
                                          fz(res=x), fl), wo, wo + 4 * D + 8 * D, "fused o+residual"))
        wg = 2 * weight_bytes("q4k", D, F)
        lst.append((lib.qgemv_q4k_fused_group, (Wb, Yb, Nb, 2, x.data_ptr(), 1, D, fz(norm=norm_w()), fl), wg,
                    wg + 8 * D + 8 * F, "fused gate/up+rmsnorm"))
        wd = weight_bytes("q4k", F, D)
        lst.append((lib.qgemv_q4k_fused, (ws[6].data_ptr(), gu[0].data_ptr(), x.data_ptr(), 1, D, F,
                                          fz(up=gu[1], res=x), fl), wd, wd + 8 * F + 8 * D, "fused down+swiglu+residual"))
    V = host[154][2]
    wv = weight_bytes("q4k", D, V)
    lst.append((lib.qgemv_q4k_fused, (mats[154].data_ptr(), x.data_ptr(), logits.data_ptr(), 1, V, D,
                                      fz(norm=norm_w()), fl), wv, wv + 8 * D + 4 * V, "fused output+rmsnorm"))
    return lst, x, logits, x0


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist
    from block_quantised_weight_gb300 import build, qgemv

    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    lib = qgemv.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    mats, desc, M = workload_spec(args.workload, args.M)
    host = gen_mats(args.workload, mats, M)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    step_wbytes = sum(weight_bytes(f, K, N) for f, K, N in mats)
    copies = 1
    if step_wbytes < 2 * l2:
        copies = int(np.ceil(2 * l2 / step_wbytes)) + 1

    # launch groups: in the decode pass q/k/v read one activation vector and
    # gate/up another, so each such set is one grouped launch (--single: one
    # launch per matrix)
    groups = pass_groups(args.workload, len(host), args.mode == "single")
    # device buffers: weights (rotated copies), x / y concatenated per pass
    xs_host = np.concatenate([host[g[0]][5].reshape(-1) for g in groups]).astype(np.float32)
    ys_len = sum(M * h[2] for h in host)
    launches = []   # per copy: list of (fn, args, wbytes, algo_bytes, label)
    keep = []
    fl = 0 if args.no_prefetch else qgemv.QG_PREFETCH_WEIGHTS
    fused = args.mode == "fused"
    if fused:
        if args.workload != "tinyllama" or M != 1:
            raise SystemExit("--mode fused runs the TinyLlama-shaped decode step at M=1")
        lst, x_dev, y_dev, xs_host = fused_step_launches(lib, qgemv, host, dev, keep)
        ys_len = y_dev.numel()
        launches.append(lst)
    else:
        x_dev = torch.from_numpy(xs_host).to(dev)
        y_dev = torch.empty(ys_len, dtype=torch.float32, device=dev)
    for c in range(0 if fused else copies):
        xo, yo = 0, 0
        lst = []
        for grp in groups:
            fmt, K = host[grp[0]][0], host[grp[0]][1]
            xp = x_dev.data_ptr() + 4 * xo
            Wp, Yp, Ns, gd = [], [], [], None
            for i in grp:
                _f, _K, N, W, grid, _x = host[i]
                Wd = torch.from_numpy(W).to(dev)
                keep.append(Wd)
                if grid is not None:
                    gd = torch.from_numpy(grid).to(dev)
                    keep.append(gd)
                Wp.append(Wd.data_ptr())
                Yp.append(y_dev.data_ptr() + 4 * yo)
                Ns.append(N)
                yo += M * N
            wb = sum(weight_bytes(fmt, K, N) for N in Ns)
            algo = wb + 4 * M * K + 4 * M * sum(Ns)
            label = f"K{K}xN" + "+".join(str(n) for n in Ns)
            if len(grp) > 1:
                Wa = (ctypes.c_void_p * len(grp))(*Wp)
                Ya = (ctypes.c_void_p * len(grp))(*Yp)
                Na = (ctypes.c_int64 * len(grp))(*Ns)
                keep.append((Wa, Ya, Na))
                if fmt == "q4k":
                    lst.append((lib.qgemv_q4k_group, (Wa, Ya, Na, len(grp), xp, M, K, fl), wb, algo, label))
                else:
                    lst.append((lib.qgemv_iq3_group, (Wa, Ya, Na, len(grp), gd.data_ptr(), xp, M, K, fl), wb, algo,
                                label))
            elif fmt == "q4k" and M >= 16:
                lst.append((lib.qgemm_q4k_batched, (Wp[0], xp, Yp[0], M, Ns[0], K), wb, algo, label))
            elif fmt == "q4k":
                lst.append((lib.qgemv_q4k_ex, (Wp[0], xp, Yp[0], M, Ns[0], K, fl), wb, algo, label))
            elif fmt == "iq3" and M >= 16:
                lst.append((lib.qgemm_iq3_batched, (Wp[0], gd.data_ptr(), xp, Yp[0], M, Ns[0], K), wb, algo, label))
            elif fmt == "iq3":
                lst.append((lib.qgemv_iq3_ex, (Wp[0], gd.data_ptr(), xp, Yp[0], M, Ns[0], K, fl), wb, algo, label))
            elif fmt == "iq3xxs":
                lst.append((lib.qgemv_iq3xxs_ex, (Wp[0], gd.data_ptr(), xp, Yp[0], M, Ns[0], K, fl), wb, algo, label))
            else:
                lst.append((lib.qgemv_codebook, (qgemv.QG_CB[fmt], Wp[0], gd.data_ptr(), xp, Yp[0], M, Ns[0], K), wb,
                            algo, label))
            xo += M * K
        if args.mode == "pass" and args.workload == "tinyllama":
            # the whole pass as one persistent launch: stage i reads its x only
            # after stage i-1 has written all of its y
            arr = (qgemv.QgStage * len(lst))()
            for i, (fn, a, wb, ab, lb) in enumerate(lst):
                st = arr[i]
                if fn == lib.qgemv_q4k_group:
                    Wa, Ya, Na, cnt, xp, _M, K, _fl = a
                    st.count = cnt
                    for j in range(cnt):
                        st.W[j], st.Y[j], st.N[j] = Wa[j], Ya[j], Na[j]
                else:
                    Wp0, xp, yp0, _M, N0, K, _fl = a
                    st.count = 1
                    st.W[0], st.Y[0], st.N[0] = Wp0, yp0, N0
                st.X = xp
                st.K = K
            sync = torch.zeros(len(lst) + 8, dtype=torch.int32, device=dev)
            keep.append((arr, sync))
            lst = [(lib.qgemv_q4k_pass, (arr, len(lst), M, sync.data_ptr()), sum(l[2] for l in lst),
                    sum(l[3] for l in lst), f"pass({len(lst)} stages)")]
        launches.append(lst)
    flat = [l for lst in launches for l in lst]

    stream = torch.cuda.Stream(device=dev)
    sh = ctypes.c_void_p(stream.cuda_stream)

    def run_pass(lst):
        for fn, a, _wb, _ab, _lb in lst:
            rc = fn(*a, sh)
            if rc != 0:
                raise RuntimeError(f"launch failed: {rc} {qgemv.strerror(rc)}")

    with torch.cuda.stream(stream):
        for _ in range(2):
            for lst in launches:
                run_pass(lst)
    torch.cuda.synchronize(dev)
    assert qgemv.qg_device_status() == 0

    # graph of one step (all copies, so one replay = `copies` passes); a second,
    # instrumented graph holds an external event pair around every launch for
    # per-launch kernel durations (the event nodes serialise the launches, so
    # it is replayed after the timed region, not inside it)
    rt = cudart()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in flat]
    for a, b in ev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    per_launch_ok = rt is not None and hasattr(ev[0][0], "cuda_event")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        cap = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for fn, a, _wb, _ab, _lb in flat:
            rc = fn(*a, cap)
            if rc != 0:
                raise RuntimeError(f"capture launch failed: {rc}")
    gi = torch.cuda.CUDAGraph()
    if per_launch_ok:
        with torch.cuda.graph(gi, stream=stream):
            cap = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            for i, (fn, a, _wb, _ab, _lb) in enumerate(flat):
                if per_launch_ok:
                    per_launch_ok = rt.cudaEventRecordWithFlags(ctypes.c_void_p(ev[i][0].cuda_event), cap, 1) == 0
                rc = fn(*a, cap)
                if rc != 0:
                    raise RuntimeError(f"capture launch failed: {rc}")
                if per_launch_ok:
                    per_launch_ok = rt.cudaEventRecordWithFlags(ctypes.c_void_p(ev[i][1].cuda_event), cap, 1) == 0
    passes_per_replay = copies

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            g.replay()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # REPEATS timed regions of exactly `steps` steps, each bracketed by a
    # barrier and a device synchronisation; the slowest rank's time of each,
    # and the median region is reported
    region_ms = []
    for _ in range(REPEATS):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(args.steps):
                g.replay()
            t1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        region_ms.append(t0.elapsed_time(t1))
    region_ms = max_over_ranks(region_ms, world, dev)
    ms_total = statistics.median(region_ms)
    durs = None
    if per_launch_ok:
        try:
            with torch.cuda.stream(stream):
                for _ in range(3):
                    gi.replay()
            torch.cuda.synchronize(dev)
            durs = [a.elapsed_time(b) for a, b in ev]
        except Exception:
            durs = None
    status = qgemv.qg_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")

    # dependent-launch floor of the step: the same chain of launches (same
    # count, grids and x lengths) doing no weight work (qg_test_chain_step)
    floor = None
    if args.workload == "tinyllama" and args.mode in ("group", "fused"):
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        ybuf = torch.empty(2 * sms * 32 + 64, dtype=torch.float32, device=dev)
        chain = []
        for grp in groups:
            K = host[grp[0]][1]
            tiles = sum((host[i][2] + 31) // 32 for i in grp)
            chain.append((K, min(tiles, 2 * sms)))
        xs_len = max(K for K, _ in chain)
        xf = torch.zeros(xs_len, dtype=torch.float32, device=dev)
        gf = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf, stream=stream):
            cap = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            for K, gx in chain:
                rc = lib.qg_test_chain_step(xf.data_ptr(), ybuf.data_ptr(), K, gx, qgemv.QG_PREFETCH_WEIGHTS, cap)
                if rc != 0:
                    raise RuntimeError(f"chain step failed: {rc}")
        with torch.cuda.stream(stream):
            for _ in range(3):
                gf.replay()
        torch.cuda.synchronize(dev)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            f0.record(stream)
            for _ in range(args.steps):
                gf.replay()
            f1.record(stream)
        torch.cuda.synchronize(dev)
        floor_ms = f0.elapsed_time(f1) / args.steps
        floor = {"ms_per_pass": round(floor_ms, 4), "launches": len(chain),
                 "note": "the same chain of programmatic dependent launches (grids min(tiles, 2 x SMs), each "
                         "reading its x) doing no weight work: the part of the step time that streaming and "
                         "decoding inside this launch chain cannot remove"}

    # e2e: host x in, host y out, every step, through the same C-ABI calls
    xs_pin = torch.from_numpy(xs_host).pin_memory()
    ys_pin = torch.empty(ys_len, dtype=torch.float32).pin_memory()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(2):
            x_dev.copy_(xs_pin, non_blocking=True)
            g.replay()
            ys_pin.copy_(y_dev, non_blocking=True)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            x_dev.copy_(xs_pin, non_blocking=True)
            g.replay()
            ys_pin.copy_(y_dev, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = e0.elapsed_time(e1)

    ms_e2e = max_over_ranks([ms_e2e], world, dev)[0]
    # the single-matrix configurations at M=1, measured in the same run (one GPU)
    per_config = None
    if world == 1 and args.workload == "tinyllama" and args.mode == "group" and not args.no_per_config:
        per_config = measure_configs(lib, qgemv, dev, stream, l2)
    clocks = sampler.stop() if sampler else None
    n_pass = args.steps * passes_per_replay
    ms_step = ms_total / n_pass
    value = job_throughput(world, step_wbytes, n_pass, ms_total)
    e2e_value = job_throughput(world, step_wbytes, n_pass, ms_e2e)

    if floor:
        floor["above_floor_ms_per_pass"] = round(ms_step - floor["ms_per_pass"], 4)
    peak, peak_kind = measured_peaks()
    # Dominant kernel (the only one in the timed region): algorithmic bytes per
    # launch / average launch duration, the duration taken from the timed
    # region on the launch stream divided by the launches in it (consecutive
    # launches overlap under programmatic dependent launch, so events around
    # each launch would serialise them).
    n_launch = len(flat) * args.steps
    algo = sum(ab for _f, _a, _wb, ab, _lb in flat)
    avg_launch_ms = ms_total / n_launch
    achieved = (algo / len(flat)) / (avg_launch_ms * 1e-3) / 1e9
    if args.mode == "pass" and args.workload == "tinyllama":
        kname = "qgemv_q4k_pass qg_gemv_pass_kernel"
    elif fused:
        kname = "qgemv_q4k_fused qg_gemv_kernel<FmtQ4KT, FUSE>"
    elif mats[0][0] == "q4k":
        kname = ("qgemm_q4k_batched qg_gemm_tc_kernel (tcgen05, bf16 weights)" if M >= 16 else
                 "qgemv_q4k qg_gemm_tc_x_kernel<Q4_K, 3> (tcgen05, x in three bf16 parts)" if M >= 5 else
                 "qgemv_q4k qg_gemv_kernel<FmtQ4KT>")
    elif mats[0][0] == "iq3":
        kname = ("qgemm_iq3_batched qg_gemm_tc_x_kernel<IQ3, 1> (tcgen05)" if M >= 16 else
                 "qgemv_iq3 qg_gemm_tc_x_kernel<IQ3, 3> (tcgen05, x in three bf16 parts)" if M >= 5 else
                 "qgemv_iq3 qg_gemv_kernel<FmtIQ3T>")
    elif mats[0][0] == "iq3xxs":
        kname = "qgemv_iq3xxs qg_gemv_kernel<FmtIQ3XXST>"
    else:
        kname = (f"qgemv_codebook qg_gemv_cb_tma_kernel<{mats[0][0].upper()}>" if mats[0][0] in ("iq4nl", "iq4xs")
                 else f"qgemv_codebook qg_gemv_cb_kernel<{mats[0][0].upper()}>")
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": profiled_traffic(args.workload, M),
            "peak_kind": f"of {peak_kind}", "kernel": kname, "launches_timed": n_launch,
            "avg_launch_us": round(1e3 * avg_launch_ms, 3), "algorithmic_bytes_per_launch": round(algo / len(flat)),
            "durations": "CUDA events on the launch stream around the timed region / launches in it"}
    # 2 <= M <= 15 on the fp32 FMA path: the arithmetic (2*M flops per weight)
    # can take longer than the weight stream, so the roofline is the lower of
    # the two ceilings; the fp32 peak is the SMs' FMA lanes (128 per SM, 2
    # flops each) at the largest SM clock sampled during the run
    fma_path = fused or mats[0][0] not in ("q4k", "iq3") or M < 5
    if fma_path and 2 <= M <= 15:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
        fp32_peak = sms * 128 * 2 * mhz * 1e6 / 1e12  # TFLOP/s
        flops = 2.0 * M * sum(K * N for _f, K, N in mats)  # per step
        tflops = flops / (ms_step * 1e-3) / 1e12
        if flops / (fp32_peak * 1e12) > step_wbytes / (peak * 1e9):  # the arithmetic takes longer
            hbm_view = {k: roof[k] for k in ("achieved", "peak", "unit", "frac", "peak_kind")}
            roof.update({"bound": "alu", "achieved": round(tflops, 2), "peak": round(fp32_peak, 1), "unit": "TFLOP/s",
                         "frac": round(tflops / fp32_peak, 4),
                         "peak_kind": f"of nominal ({sms} SMs x 128 fp32 FMA lanes x 2 flop at {mhz:.0f} MHz)",
                         "hbm_view": hbm_view})
    if durs:
        kern_ms = sum(durs)
        by_shape = {}
        for (fn, a, wb, ab, key), d in zip(flat, durs):
            e = by_shape.setdefault(key, [0, 0.0, 0])
            e[0] += 1
            e[1] += d
            e[2] += ab
        roof["serialised"] = {
            "note": "events around every launch in a replay right after the timed region (launches serialised)",
            "kernel_ms_per_pass": round(kern_ms / passes_per_replay, 4),
            "per_shape": {k: {"launches": n, "us_per_launch": round(1e3 * t / n, 2),
                              "GBps": round(b / (t * 1e-3) / 1e9, 1)} for k, (n, t, b) in by_shape.items()}}
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy; shapes of the pages' models)",
        "config": {"workload": desc, "M": M, "weight_bytes_per_step": step_wbytes,
                   "launches_per_step": len(flat) // copies,
                   "l2": ("inputs larger than L2" if copies == 1 else
                          f"rotates {copies} weight copies (> 2x L2)"),
                   "graph": "CUDA graph of the step, replayed", "parallelism": f"replicas x{world}",
                   "launch": ("one persistent cooperative launch per pass (qgemv_q4k_pass); stage i reads x only "
                              "after every CTA finished stage i-1; weights of later stages stream meanwhile"
                              if args.mode == "pass" and args.workload == "tinyllama" else
                              "decode step with its data flow on the device: fused RMSNorm / SwiGLU prologues "
                              "and residual epilogues, each GEMV reading the previous one's output "
                              "(programmatic dependent launch)" if fused else
                              "stream-ordered" if args.no_prefetch else
                              "programmatic dependent launch: each GEMV streams its first weight tiles while "
                              "the previous one finishes and waits for it before reading x")},
        "tokens_per_s_equiv": round(world * 1000.0 / ms_step, 1),
        "gemv_per_s": round(world * len(mats) * 1000.0 / ms_step, 1),
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": int(xs_host.nbytes),
                "d2h_bytes_per_step": int(4 * ys_len),
                "note": ("pinned host x (the embedding row) -> device, graph of C-ABI launches, device logits -> "
                         "pinned host, every step" if fused else
                         "pinned host x -> device, graph of C-ABI launches, device y -> pinned host, every step")},
        "repeats": {"n": REPEATS, "statistic": "median",
                    "ms_per_step_each": [round(r / n_pass, 4) for r in region_ms]},
        "gpu_launches": sum(kernel_launches(lib, fn, a, M) for fn, a, _wb, _ab, _lb in flat) * args.steps,
        "mode": args.mode,
        "latency_floor": floor,
        "roofline": roof,
        "per_config": per_config,
        "clocks": clocks,
    }


# ------------------------------------------------------------------ per-config block
REPEATS = 5
PER_CONFIG = ("q4k_c0", "iq3_c2", "q4k_c4a", "q4k_c4b", "iq3_c4a", "iq3_c4b")


def measure_configs(lib, qgemv, dev, stream, l2, min_region_ms=200.0):
    """The single-matrix M=1 configurations, each timed as REPEATS regions of
    at least min_region_ms (a CUDA graph of launches rotating over weight
    copies that together exceed 2x L2, replayed), median region reported."""
    import numpy as np
    import torch
    peak, peak_kind = measured_peaks()
    out = []
    for name in PER_CONFIG:
        mats, desc, M = workload_spec(name, 1)
        fmt, K, N = mats[0]
        host = gen_mats(name, mats, 1)
        wb = weight_bytes(fmt, K, N)
        copies = int(np.ceil(2 * l2 / wb)) + 1 if wb < 2 * l2 else 1
        _f, _K, _N, W, grid, x = host[0]
        xd = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        yd = torch.empty((1, N), dtype=torch.float32, device=dev)
        gd = torch.from_numpy(grid).to(dev) if grid is not None else None
        Wds = [torch.from_numpy(W).to(dev) for _ in range(copies)]
        fl = qgemv.QG_PREFETCH_WEIGHTS

        def launch(Wd, s):
            if fmt == "q4k":
                return lib.qgemv_q4k_ex(Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), 1, N, K, fl, s)
            return lib.qgemv_iq3_ex(Wd.data_ptr(), gd.data_ptr(), xd.data_ptr(), yd.data_ptr(), 1, N, K, fl, s)

        per_graph = max(copies, 64 // copies * copies)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            cap = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            for i in range(per_graph):
                if launch(Wds[i % copies], cap) != 0:
                    raise RuntimeError(f"{name}: capture launch failed")
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        replays = max(1, int(np.ceil(min_region_ms / max(e0.elapsed_time(e1), 1e-3))))
        regions = []
        for _ in range(REPEATS):
            torch.cuda.synchronize(dev)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(replays):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize(dev)
            regions.append(e0.elapsed_time(e1))
        status = qgemv.qg_device_status()
        if status != 0:
            raise RuntimeError(f"{name}: device status {status}")
        ms = statistics.median(regions) / (replays * per_graph)
        gbps = wb / (ms * 1e-3) / 1e9
        out.append({"workload": desc, "fmt": fmt, "K": K, "N": N, "M": 1, "ms": round(ms, 5),
                    "GBps": round(gbps, 1), "roofline_frac": round(gbps / peak, 4),
                    "peak": peak, "peak_kind": f"of {peak_kind}",
                    "tokens_per_s_equiv": round(1000.0 / ms, 1), "gemv_per_s": round(1000.0 / ms, 1),
                    "launches_per_region": replays * per_graph,
                    "region_ms_each": [round(r, 2) for r in regions], "weight_copies": copies})
        del Wds, g
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ oracle arm
def oracle_sample_rate(workload, M, budget_s, threads=None):
    """Oracle weight GB/s on a bounded sample of the workload (full rows)."""
    import numpy as np

    import oracle
    mats, _desc, M = workload_spec(workload, M)
    host = gen_mats(workload, mats[:7], M) if workload == "tinyllama" else gen_mats(workload, mats, M)
    done_bytes, t_used, n = 0, 0.0, 0
    nt = oracle.max_threads() if threads is None else threads
    rows_cap = []
    for fmt, K, N, W, grid, x in host:
        rows_cap.append(min(N, max(64, int(4e6 // K))))
    t_start = time.perf_counter()
    while t_used < budget_s:
        for (fmt, K, N, W, grid, x), nr in zip(host, rows_cap):
            rows = np.arange(nr)
            t0 = time.perf_counter()
            if fmt == "q4k":
                oracle.gemv_q4k(W[:nr], x, rows=rows, nthreads=nt)
            elif fmt == "iq3":
                oracle.gemv_iq3(W[:nr], grid, x, rows=rows, nthreads=nt)
            elif fmt == "iq3xxs":
                oracle.gemv_iq3xxs(W[:nr], grid, x, rows=rows, nthreads=nt)
            else:
                oracle.gemv_cb(fmt, W[:nr], grid, x, rows=rows, nthreads=nt)
            t_used += time.perf_counter() - t0
            done_bytes += weight_bytes(fmt, K, nr)
            n += 1
            if t_used >= budget_s:
                break
    sample = ("first 7 matrices of the pass (layer 0), first rows of each" if workload == "tinyllama"
              else "first rows of the matrix") + f", {n} matrix calls, {done_bytes / 1e6:.1f} MB"
    return done_bytes / t_used / 1e9, nt, sample


def run_reference(args, rank, world):
    if rank != 0:
        return None
    mats, desc, M = workload_spec(args.workload, args.M)
    step_budget = 2.0
    for _ in range(args.warmup):
        oracle_sample_rate(args.workload, args.M, 0.2)
    t0 = time.perf_counter()
    rates, nt, sample = [], 1, ""
    for _ in range(args.steps):
        r, nt, sample = oracle_sample_rate(args.workload, args.M, step_budget)
        rates.append(r)
    wall = time.perf_counter() - t0
    value = statistics.median(rates)
    step_wbytes = sum(weight_bytes(f, K, N) for f, K, N in mats)
    ms_step = step_wbytes / (value * 1e9) * 1e3
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "M": M, "weight_bytes_per_step": step_wbytes},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": nt, "kind": "oracle",
                         "sample": sample + f"; {step_budget:.0f} s of oracle time per step"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 1),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="tinyllama")
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--cpu-baseline-s", type=float, default=12.0)
    ap.add_argument("--no-prefetch", action="store_true", help="plain stream-ordered launches")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the single-matrix M=1 configurations measured after the decode pass")
    ap.add_argument("--mode", choices=["pass", "group", "single", "fused"], default="group",
                    help="decode pass as one persistent launch (pass), one launch per q/k/v or gate/up group "
                         "(group), one launch per matrix (single), or the decode step with fused RMSNorm / "
                         "SwiGLU / residual and its data flow on the device (fused)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        r, nt, sample = oracle_sample_rate(args.workload, args.M, args.cpu_baseline_s)
        out["cpu_baseline"] = {"value": round(r, 3), "unit": "GB/s", "cores": nt, "kind": "oracle",
                               "sample": sample}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
