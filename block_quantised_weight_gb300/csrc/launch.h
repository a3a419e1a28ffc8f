// Host-side launchers shared between the translation units of libqgemv.
// Arguments are validated by the C-ABI layer (api.cu) before these run.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qgemv.h"

namespace qg {

// The CUDA error behind the calling host thread's last QG_ECUDA (0 when the
// failing step was not a CUDA runtime call, e.g. a tensor-map encoding).
inline thread_local int t_last_cuda_error = 0;
inline int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return QG_ECUDA;
}
// Status of the launch just made on this thread: QG_OK or QG_ECUDA (recorded).
inline int launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

int launch_gemv_q4k(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t s,
                    unsigned* status, unsigned flags);
int launch_gemv_iq3(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                    cudaStream_t s, unsigned* status, unsigned flags);
struct Fuse;
int launch_group_q4k(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const float* X, int M,
                     int64_t K, cudaStream_t s, unsigned* status, unsigned flags, const Fuse* fz);
// RMSNorm / SwiGLU prologue (M <= 4) and residual epilogue, see gemv_kernel.cuh's Fuse
int launch_group_q4k_fused(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const float* X,
                           int M, int64_t K, cudaStream_t s, unsigned* status, unsigned flags, const Fuse& fz);
int launch_gemv_iq3xxs(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                       cudaStream_t s, unsigned* status, unsigned flags);
int launch_dequant_iq3xxs(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K, cudaStream_t s);
int launch_group_iq3(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const uint8_t* grid,
                     const float* X, int M, int64_t K, cudaStream_t s, unsigned* status, unsigned flags);
// page 3's codebook formats (QG_CB_*)
int cb_unit_bytes(int format);
int launch_gemv_cb(int format, const uint8_t* W, const void* book, const float* X, float* Y, int M, int64_t N,
                   int64_t K, cudaStream_t s, unsigned* status);
int launch_dequant_cb(int format, const uint8_t* W, const void* book, float* out, int64_t N, int64_t K,
                      cudaStream_t s);
int launch_chain_step(const float* X, float* Y, int64_t K, int grid, unsigned flags, cudaStream_t s);
int launch_pass_q4k(const qg_stage* stages, int nstages, int M, unsigned* sync, cudaStream_t s, unsigned* status);
int launch_dequant_q4k(const uint8_t* W, float* out, int64_t N, int64_t K, cudaStream_t s);
int launch_dequant_iq3(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K, cudaStream_t s);
// tcgen05 paths, 16 <= M <= 32: Q4_K weights rounded to bf16; IQ3 weights
// exact (signed grid bytes, sub-block factors applied after the MMA), x
// rounded to bf16
int launch_gemm_q4k_tc(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t s,
                       unsigned* status);
int launch_gemm_iq3_tc(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                       cudaStream_t s, unsigned* status);
// tcgen05 IQ3 with x split exactly into three bf16 parts, 1 <= M <= 10:
// exact products, fp32 accumulation (the fp32 FMA path's bar)
int launch_gemm_iq3_tc3(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                        cudaStream_t s, unsigned* status);
// tcgen05 Q4_K the same way, 1 <= M <= 10: A = q - c (the offset of the FMA
// path's exact factoring), a * sum - r * sum(x) per sub-block afterwards
int launch_gemm_q4k_tc3(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t s,
                        unsigned* status);

}  // namespace qg
