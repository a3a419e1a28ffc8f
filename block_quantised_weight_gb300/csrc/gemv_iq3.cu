// IQ3 GEMV launcher, page 4's block order.  Dispatch: launch_iq3.cuh.
#include "launch_iq3.cuh"

namespace qg {

int launch_group_iq3(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const uint8_t* grid,
                     const float* X, int M, int64_t K, cudaStream_t s, unsigned* status, unsigned flags) {
    return launch_group_iq3_t<FmtIQ3T>(W, Y, N, count, grid, X, M, K, s, status, flags);
}

int launch_gemv_iq3(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                    cudaStream_t s, unsigned* status, unsigned flags) {
    return launch_group_iq3(&W, &Y, &N, 1, grid, X, M, K, s, status, flags);
}

}  // namespace qg
