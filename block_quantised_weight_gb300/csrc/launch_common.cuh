// Host-side helpers shared by the GEMV launchers.
#pragma once
#include <algorithm>
#include <atomic>

#include "gemv_kernel.cuh"
#include "launch.h"
#include "tensor_map.h"

namespace qg {

inline int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    return dev;
}

// Per-device values computed on first use.  Host threads may race to fill a
// slot; they all store the same value, and atomics keep that well defined.
inline int sm_count(int dev) {
    static std::atomic<int> cache[64];
    if (dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Launch qg_gemv_kernel<F, MT, RG, MINB, FUSE> over `count` matrices that
// share X (token offset m0 already applied to X; Y[i] + m0*N[i] here): MINB
// CTAs per SM, as many pipeline stages as fit in the per-CTA share of shared
// memory.
template <class F, int MT, int RG, int MINB, int FUSE = 0>
int launch_gemv(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, int m0, const uint8_t* grid,
                const float* X, int M, int64_t K, cudaStream_t s, unsigned* status, int dev, unsigned flags,
                int csize = 1, const Fuse* fz = nullptr) {
    static std::atomic<bool> attr_done[64];
    constexpr int kThreads = RG * F::kCols * F::kWPC * 32 + 32;  // consumer warps + the producer
    const int budget = std::min(kSmemPerCTA, kSmemPerSM / MINB - kSmemReserve);
    const Layout L1 = make_layout(F::kIQ3, MT, F::kXH, RG, 1, F::kRowStride, F::kCols, FUSE, F::kWPC);
    const int stages_fit = std::min(kMaxStages, (budget - L1.stage0) / L1.stage_bytes);
    if (stages_fit < 2) return QG_EINVAL;
    auto kern = qg_gemv_kernel<F, MT, RG, MINB, FUSE>;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        const Layout Lmax = make_layout(F::kIQ3, MT, F::kXH, RG, stages_fit, F::kRowStride, F::kCols, FUSE, F::kWPC);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lmax.total) != cudaSuccess)
            return qg::cuda_fail(cudaGetLastError());
        attr_done[dev].store(true, std::memory_order_release);
    }
    // prologue operands and residuals (token offset m0 applied like X, Y)
    Fuse Fz = {};
    if (fz) {
        Fz = *fz;
        if (Fz.up) Fz.up += static_cast<int64_t>(m0) * K;
        for (int i = 0; i < count; ++i)
            if (Fz.R[i]) Fz.R[i] += static_cast<int64_t>(m0) * N[i];
    }
    for (int i = count; i < kMaxGroup; ++i) Fz.R[i] = nullptr;
    Group G = {};
    G.count = count;
    G.tile0[0] = 0;
    for (int i = 0; i < count; ++i) {
        G.W[i] = W[i];
        G.Y[i] = Y[i] + static_cast<int64_t>(m0) * N[i];
        G.N[i] = N[i];
        G.tile0[i + 1] = G.tile0[i] + (N[i] + RG * kRows - 1) / (RG * kRows);
    }
    TMaps T = {};
    {
        const uint64_t pitch = static_cast<uint64_t>(K / 256) * F::kBytes;
        for (int i = 0; i < count; ++i)
            if (!encode_byte_rows(&T.m[i], W[i], pitch, static_cast<uint64_t>(N[i]), F::kBoxBytes, RG * kRows))
                return qg::cuda_fail(cudaGetLastError());
    }
    if (F::kXH == kXHalf && !encode_x_halves(&T.xm, X, static_cast<uint64_t>(M) * static_cast<uint64_t>(K / 128))) return qg::cuda_fail(cudaGetLastError());
    const int64_t ntiles = G.tile0[count];
    const int sms = sm_count(dev);
    if (sms <= 0) return qg::cuda_fail(cudaGetLastError());
    // csize > 1: one CTA per (tile, K chunk), the chunks of a tile in one
    // cluster (the caller checks that the grid fits one wave).
    const int grid_x = csize > 1 ? static_cast<int>(ntiles * csize)
                                 : static_cast<int>(std::min<int64_t>(ntiles, static_cast<int64_t>(sms) * MINB));
    // A ring deeper than a CTA's units only takes shared memory from the CTAs
    // of the next launch, which could otherwise become resident early and
    // start their weight stream: at most one stage per unit.
    const int64_t nch = (K / 256 + F::kCols - 1) / F::kCols;
    const int64_t units = csize > 1 ? 1 : (ntiles + grid_x - 1) / grid_x * nch;
    const int stages = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(stages_fit, units)));
    const Layout L = make_layout(F::kIQ3, MT, F::kXH, RG, stages, F::kRowStride, F::kCols, FUSE, F::kWPC);
    const int kflags = ((flags & QG_PREFETCH_WEIGHTS) ? kFlagPrefetchWeights : 0) |
                       (csize > 1 ? csize << kFlagClusterShift : 0);
    if (!(flags & QG_PREFETCH_WEIGHTS) && csize <= 1) {
        kern<<<grid_x, kThreads, L.total, s>>>(G, T, Fz, grid, X, M, K, stages, status, kflags);
        return launch_status();
    }
    // programmatic dependent launch (this grid may start before the previous
    // kernel in the stream finishes; the kernel waits before reading x) and/or
    // a cluster launch
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (flags & QG_PREFETCH_WEIGHTS) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (csize > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = csize;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kern, G, T, Fz, grid, X, M, K, stages, status, kflags) != cudaSuccess)
        return qg::cuda_fail(cudaGetLastError());
    return launch_status();
}

}  // namespace qg
