// Q4_K GEMV with a fused prologue on x: RMSNorm (page 2 "Candle",
// RmsNorm::forward) or SwiGLU (page 2 "Candle", Block::forward:
// silu(gate) * up); residual epilogues ride along.  Dispatch: launch_q4k.cuh.
#include "launch_q4k.cuh"

namespace qg {

int launch_group_q4k_fused(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const float* X,
                           int M, int64_t K, cudaStream_t s, unsigned* status, unsigned flags, const Fuse& fz) {
    if (fz.g) return launch_group_q4k_t<kFuseNorm>(W, Y, N, count, X, M, K, s, status, flags, &fz);
    if (fz.up) return launch_group_q4k_t<kFuseSwiGLU>(W, Y, N, count, X, M, K, s, status, flags, &fz);
    return launch_group_q4k_t<0>(W, Y, N, count, X, M, K, s, status, flags, &fz);
}

}  // namespace qg
