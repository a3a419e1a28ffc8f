// Test-only: the dependent-launch floor of a decode step.  One launch of
// qg_chain_step_kernel does what every GEMV of the step must do on the
// dependency chain and nothing else: let the next launch start
// (griddepcontrol.launch_dependents), wait for the previous one
// (griddepcontrol.wait), read the activation vector x and write 32 outputs
// per CTA.  A chain of these with the grids of the step's GEMVs measures the
// part of the step time that no weight streaming or decoding inside the
// chain can remove.
#include "launch_common.cuh"

namespace qg {

__global__ void __launch_bounds__(288) qg_chain_step_kernel(const float* __restrict__ X, float* __restrict__ Y,
                                                         int64_t K) {
    grid_launch_dependents();
    grid_dependency_wait();
    float acc = 0.f;
    for (int64_t i = threadIdx.x; i < K / 4; i += blockDim.x) {
        const float4 v = reinterpret_cast<const float4*>(X)[i];
        acc += (v.x + v.y) + (v.z + v.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (threadIdx.x < 32) Y[static_cast<int64_t>(blockIdx.x) * 32 + threadIdx.x] = acc;
}

int launch_chain_step(const float* X, float* Y, int64_t K, int grid, unsigned flags, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(288);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & QG_PREFETCH_WEIGHTS) ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, qg_chain_step_kernel, X, Y, K) != cudaSuccess) return qg::cuda_fail(cudaGetLastError());
    return launch_status();
}

}  // namespace qg
