// tcgen05 (bf16, fp32 accumulation in tensor memory) path for M >= 16.
#include "launch.h"

namespace qg {

int launch_gemm_q4k_tc(const uint8_t*, const float*, float*, int, int64_t, int64_t, cudaStream_t, unsigned*) {
    return QG_EINVAL;  // not built yet
}

}  // namespace qg
