// IQ3_XXS GEMV launcher: page 3's byte order for the 98-byte IQ3 block (d
// first, eff = d*(0.5+s)*0.5 times the raw codebook entry).  Dispatch:
// launch_iq3.cuh.
#include "launch_iq3.cuh"

namespace qg {

int launch_gemv_iq3xxs(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                       cudaStream_t s, unsigned* status, unsigned flags) {
    return launch_group_iq3_t<FmtIQ3XXST>(&W, &Y, &N, 1, grid, X, M, K, s, status, flags);
}

}  // namespace qg
