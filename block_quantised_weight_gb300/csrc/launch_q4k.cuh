// Q4_K GEMV dispatch (fp32 FMA path), shared by the plain and the fused
// translation units.  Kernel: gemv_kernel.cuh.
#pragma once
#include "launch_common.cuh"

namespace qg {

// count matrices sharing X; M is split into token groups, each streaming W
// once: from 5 tokens without prologue or residual the tcgen05 kernel of
// gemm_tc.cu (groups of 5 to 10, x in three exact bf16 parts, the FMA
// path's offset factoring), otherwise groups of at most 4 on the fp32 FMA
// kernels.  FUSE != 0 (a prologue on x) needs M <= 4: the staged-x kernels
// apply it.  fz may carry residuals with any FUSE.
template <int FUSE>
int launch_group_q4k_t(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const float* X, int M,
                       int64_t K, cudaStream_t s, unsigned* status, unsigned flags, const Fuse* fz) {
    const int dev = current_device();
    if (dev < 0) return qg::cuda_fail(cudaGetLastError());
    if (FUSE != 0 && M > 4) return QG_EINVAL;
    // Launches with at most one 32-row tile per SM are latency-bound: run them
    // one CTA per SM.  A unit's decode is bound by the SM's issue rate either
    // way, but the prologue kernels (RMSNorm, SwiGLU) measure faster with 16
    // consumer warps, two per column (FmtQ4KT2).
    int64_t tiles = 0;
    for (int i = 0; i < count; ++i) tiles += (N[i] + kRows - 1) / kRows;
    const int sms = sm_count(dev);
    const bool few_tiles = tiles <= sms;
    // ... and when the tiles' K chunks fit one wave of two CTAs per SM, each
    // chunk gets its own CTA, the chunks of a tile forming one cluster.
    const int64_t nchunks = (K / 256 + kCols - 1) / kCols;
    const int csize = (nchunks > 1 && nchunks <= kMaxCluster && tiles * nchunks <= 2 * sms) ? static_cast<int>(nchunks) : 1;
    bool residual = false;
    if (fz)
        for (int i = 0; i < count; ++i) residual = residual || fz->R[i] != nullptr;
    if (FUSE == 0 && !residual && M >= 5) {
        // 5 or more tokens: the tensor cores, x split exactly into three bf16
        // parts (gemm_tc.cu), in ceil(M / 10) balanced token groups of 5 to
        // 10, one pass over W each
        const int ng = (M + 9) / 10;
        for (int g = 0; g < ng; ++g) {
            const int m0 = M * g / ng, m1 = M * (g + 1) / ng;
            for (int i = 0; i < count; ++i) {
                const int rc = launch_gemm_q4k_tc3(W[i], X + static_cast<int64_t>(m0) * K,
                                                   Y[i] + static_cast<int64_t>(m0) * N[i], m1 - m0, N[i], K, s, status);
                if (rc != QG_OK) return rc;
            }
        }
        return QG_OK;
    }
    for (int m0 = 0; m0 < M;) {
        const float* Xg = X + static_cast<int64_t>(m0) * K;
        const int mg = std::min(4, M - m0);
        int rc;
        if (mg == 1 && csize > 1)
            rc = launch_gemv<FmtQ4KT, 1, 1, 2, FUSE>(W, Y, N, count, m0, nullptr, Xg, mg, K, s, status, dev,
                                                           flags, csize, fz);
        else if (mg == 1 && few_tiles && FUSE != 0)  // prologue kernels: two warps per column stage x in parallel
            rc = launch_gemv<FmtQ4KT2, 1, 1, 1, FUSE>(W, Y, N, count, m0, nullptr, Xg, mg, K, s, status, dev,
                                                            flags, 1, fz);
        else if (mg == 1 && few_tiles)  // one CTA per SM: a deeper ring prefetches every unit of a tile
            rc = launch_gemv<FmtQ4KT, 1, 1, 1, FUSE>(W, Y, N, count, m0, nullptr, Xg, mg, K, s, status, dev,
                                                           flags, 1, fz);
        else if (mg == 1)
            rc = launch_gemv<FmtQ4KT, 1, 1, 2, FUSE>(W, Y, N, count, m0, nullptr, Xg, mg, K, s, status, dev,
                                                           flags, 1, fz);
        else if (mg == 2)  // prologue operands double a stage's x area: one CTA per SM then
            rc = launch_gemv<FmtQ4KT, 2, 1, FUSE == 0 ? 2 : 1, FUSE>(W, Y, N, count, m0, nullptr, Xg, mg, K, s,
                                                                           status, dev, flags, 1, fz);
        else
            rc = launch_gemv<FmtQ4KT, 4, 1, 1, FUSE>(W, Y, N, count, m0, nullptr, Xg, mg, K, s, status, dev,
                                                           flags, 1, fz);
        if (rc != QG_OK) return rc;
        m0 += mg;
    }
    return QG_OK;
}

}  // namespace qg
