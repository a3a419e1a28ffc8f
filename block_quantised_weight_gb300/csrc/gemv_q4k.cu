// Q4_K GEMV launcher (fp32 FMA path), no prologue.  Dispatch: launch_q4k.cuh.
#include "launch_q4k.cuh"

namespace qg {

int launch_group_q4k(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const float* X, int M,
                     int64_t K, cudaStream_t s, unsigned* status, unsigned flags, const Fuse* fz) {
    return launch_group_q4k_t<0>(W, Y, N, count, X, M, K, s, status, flags, fz);
}

int launch_gemv_q4k(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t s,
                    unsigned* status, unsigned flags) {
    return launch_group_q4k(&W, &Y, &N, 1, X, M, K, s, status, flags, nullptr);
}

}  // namespace qg
