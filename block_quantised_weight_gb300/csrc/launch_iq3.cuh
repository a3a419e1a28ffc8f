// IQ3 GEMV dispatch for both block orders (page 4's and page 3's IQ3_XXS),
// shared by their translation units.  Kernel: gemv_kernel.cuh (fp32 FMA);
// rows whose byte offsets are not 16-byte aligned take the byte-addressed
// kernel below; page 4's order from 5 tokens the tcgen05 kernel of
// gemm_tc.cu with x in three exact bf16 parts.
#pragma once
#include <type_traits>
#include "launch_common.cuh"

namespace qg {


// ------------------------------------------------ IQ3 rows not 16-byte aligned
// When K/256 is not a multiple of 8 the 98-byte rows do not start on 16-byte
// boundaries, which bulk copies require.  This path reads bytes straight
// from global memory: one warp per row, lanes over super-blocks, the grid
// staged in smem.  Correct for every K % 256 == 0; not tuned.
template <class F>
__global__ void __launch_bounds__(256)
    qg_gemv_iq3_bytes_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ grid, const float* __restrict__ X,
                          float* __restrict__ Y, int M, int64_t N, int64_t K) {
    __shared__ uint32_t g[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) g[i] = *reinterpret_cast<const uint32_t*>(grid + 4 * i);
    __syncthreads();
    const int nb = static_cast<int>(K / 256);
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < N; row += warps) {
        float acc[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) acc[m] = 0.f;
        for (int b = lane; b < nb; b += 32) {
            const uint8_t* blk = W + (row * nb + b) * 98;
            const float d = h2f(static_cast<uint32_t>(blk[F::kDOff]) | (static_cast<uint32_t>(blk[F::kDOff + 1]) << 8));
            for (int ib = 0; ib < 8; ++ib) {
                const uint8_t* wp = blk + F::kWordOff + 4 * ib;
                const uint32_t sw = static_cast<uint32_t>(wp[0]) | (static_cast<uint32_t>(wp[1]) << 8) |
                                    (static_cast<uint32_t>(wp[2]) << 16) | (static_cast<uint32_t>(wp[3]) << 24);
                const float db = d * (static_cast<float>(sw >> 28) + 0.5f) * F::kDbScale;
                float dot[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) dot[m] = 0.f;
                for (int t = 0; t < 32; ++t) {
                    const int l = t >> 3, j = t & 7;
                    const uint32_t seven = (sw >> (7 * l)) & 0x7Fu;
                    const uint32_t neg = j < 7 ? (seven >> j) & 1u : (__popc(seven) & 1u);
                    const float mag = byte_f(g[blk[F::kIdxOff + 8 * ib + (t >> 2)]], t & 3);
                    const float wv = neg ? -mag : mag;
                    const int64_t k = static_cast<int64_t>(b) * 256 + 32 * ib + t;
#pragma unroll
                    for (int m = 0; m < 8; ++m)
                        if (m < M) dot[m] = fmaf(wv, X[m * K + k], dot[m]);
                }
#pragma unroll
                for (int m = 0; m < 8; ++m) acc[m] = fmaf(db, dot[m], acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            float v = acc[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0 && m < M) Y[m * N + row] = v;
        }
    }
}

template <class F>
int launch_group_iq3_t(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const uint8_t* grid,
                       const float* X, int M, int64_t K, cudaStream_t s, unsigned* status, unsigned flags) {
    const int dev = current_device();
    if (dev < 0) return qg::cuda_fail(cudaGetLastError());
    if ((K / 256) % 8 != 0) {
        // rows not 16-byte aligned: the byte-addressed kernel, up to 8 tokens per pass
        const int sms = sm_count(dev);
        if (sms <= 0) return qg::cuda_fail(cudaGetLastError());
        for (int m0 = 0; m0 < M; m0 += 8) {
            const int mg = std::min(8, M - m0);
            for (int i = 0; i < count; ++i) {
                const int64_t blocks = std::min<int64_t>((N[i] + 7) / 8, static_cast<int64_t>(sms) * 8);
                qg_gemv_iq3_bytes_kernel<F><<<static_cast<int>(blocks), 256, 0, s>>>(
                    W[i], grid, X + static_cast<int64_t>(m0) * K, Y[i] + m0 * N[i], mg, N[i], K);
                if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) return qg::cuda_fail(e);
            }
        }
        return QG_OK;
    }
    if constexpr (std::is_same<F, FmtIQ3T>::value) {
        if (M >= 5) {
            // 5 or more tokens: the tensor cores, x split exactly into three
            // bf16 parts (gemm_tc.cu), in ceil(M / 10) balanced token groups
            // of 5 to 10, one pass over W each
            const int ng = (M + 9) / 10;
            for (int g = 0; g < ng; ++g) {
                const int m0 = M * g / ng, m1 = M * (g + 1) / ng;
                for (int i = 0; i < count; ++i) {
                    const int rc = launch_gemm_iq3_tc3(W[i], grid, X + static_cast<int64_t>(m0) * K,
                                                       Y[i] + static_cast<int64_t>(m0) * N[i], m1 - m0, N[i], K, s,
                                                       status);
                    if (rc != QG_OK) return rc;
                }
            }
            return QG_OK;
        }
    }
    // groups of at most 4 tokens (the two-row decode with x staged; beyond
    // one token, one 32-row tile per CTA, so that two stages of the group's
    // x fit beside the tables)
    for (int m0 = 0; m0 < M; m0 += 4) {
        const int mg = std::min(4, M - m0);
        const float* Xg = X + static_cast<int64_t>(m0) * K;
        const int rc = mg == 1   ? launch_gemv<F, 1, 2, 1>(W, Y, N, count, m0, grid, Xg, mg, K, s, status, dev, flags)
                       : mg == 2 ? launch_gemv<F, 2, 1, 1>(W, Y, N, count, m0, grid, Xg, mg, K, s, status, dev, flags)
                                 : launch_gemv<F, 4, 1, 1>(W, Y, N, count, m0, grid, Xg, mg, K, s, status, dev, flags);
        if (rc != QG_OK) return rc;
    }
    return QG_OK;
}

}  // namespace qg
