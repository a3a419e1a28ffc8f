// Host-side construction of TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry-point query: no link against libcuda).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace qg {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    // The encoder is a driver call and needs a context current on this host
    // thread; the runtime binds one lazily, so a thread whose first CUDA call
    // is ours (cudaGetDevice does not bind) would fail.  A runtime no-op that
    // initialises binds the device's primary context, once per thread.
    static thread_local bool bound = false;
    if (!bound) {
        if (cudaFree(nullptr) != cudaSuccess) return nullptr;
        bound = true;
    }
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};  // racing threads store the same value
    PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_relaxed);
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cached.store(fn, std::memory_order_relaxed);
    }
    return fn;
}

// A quantised matrix viewed as bytes [rows][pitch]; box = box_bytes x
// box_rows, no swizzle, reads outside the matrix fill zeros.  pitch and the
// base address must be multiples of 16.  Returns false if encoding fails.
inline bool encode_byte_rows(CUtensorMap* map, const uint8_t* base, uint64_t pitch, uint64_t rows,
                             uint32_t box_bytes, uint32_t box_rows) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    const cuuint64_t gdim[2] = {pitch, rows};
    const cuuint64_t gstride[1] = {pitch};
    const cuuint32_t box[2] = {box_bytes, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activations X [M][K] fp32 viewed as rows of 128 floats ([M*K/128][128]);
// box = 132 floats x 16 rows.  The 4 floats past each 128-float row lie
// outside the tensor and arrive as zeros, so one box lands as 16 row halves
// 528 bytes apart: the padded per-column x layout of the GEMV stages.
// X must be 16-byte aligned and K a multiple of 256.
inline bool encode_x_halves(CUtensorMap* map, const float* X, uint64_t rows) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    const cuuint64_t gdim[2] = {128, rows};
    const cuuint64_t gstride[1] = {512};
    const cuuint32_t box[2] = {132, 16};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(X), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qg
