// Test-only dequantisation kernels (bit-exact with the pages' decode order).
#include "launch_common.cuh"

namespace qg {

// ------------------------------------------------ test-only dequantisation
// Bit-exact with the pages' fp32 evaluation order: the products and the
// difference are rounded separately (no FMA contraction).
__global__ void qg_dequant_q4k_kernel(const uint8_t* __restrict__ W, float* __restrict__ out, int64_t nblocks) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // (block, group g)
    if (i >= nblocks * 4) return;
    const int64_t bi = i >> 2;
    const int g = static_cast<int>(i & 3);
    const uint8_t* blk = W + bi * 144;
    const uint4 h = *reinterpret_cast<const uint4*>(blk);
    const float d = h2f(h.x), dmin = h2f(h.x >> 16);
    uint32_t sc03, mn03, sc47, mn47;
    q4k_scale_min_words(h.y, h.z, h.w, sc03, mn03, sc47, mn47);
    const uint32_t scw = g < 2 ? sc03 : sc47, mnw = g < 2 ? mn03 : mn47;
    const float a_lo = __fmul_rn(d, byte_f(scw, (2 * g) & 3)), b_lo = __fmul_rn(dmin, byte_f(mnw, (2 * g) & 3));
    const float a_hi = __fmul_rn(d, byte_f(scw, (2 * g + 1) & 3)), b_hi = __fmul_rn(dmin, byte_f(mnw, (2 * g + 1) & 3));
    float* o = out + bi * 256 + 64 * g;
    for (int l = 0; l < 32; ++l) {
        const uint32_t q = blk[16 + 32 * g + l];
        o[l] = __fsub_rn(__fmul_rn(a_lo, static_cast<float>(q & 15u)), b_lo);
        o[32 + l] = __fsub_rn(__fmul_rn(a_hi, static_cast<float>(q >> 4)), b_hi);
    }
}

// Both IQ3 orders (FmtIQ3T: page 4; FmtIQ3XXST: page 3): every value has at
// most 24 significant bits, so any evaluation order gives the exact value.
template <class F>
__global__ void qg_dequant_iq3_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ grid,
                                   float* __restrict__ out, int64_t nblocks) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // (block, sub-block)
    if (i >= nblocks * 8) return;
    const int64_t bi = i >> 3;
    const int ib = static_cast<int>(i & 7);
    const uint8_t* blk = W + bi * 98;
    const float d = h2f(static_cast<uint32_t>(blk[F::kDOff]) | (static_cast<uint32_t>(blk[F::kDOff + 1]) << 8));
    const uint8_t* wp = blk + F::kWordOff + 4 * ib;
    const uint32_t sw = static_cast<uint32_t>(wp[0]) | (static_cast<uint32_t>(wp[1]) << 8) |
                        (static_cast<uint32_t>(wp[2]) << 16) | (static_cast<uint32_t>(wp[3]) << 24);
    const float db = __fmul_rn(__fmul_rn(d, __fadd_rn(0.5f, static_cast<float>(sw >> 28))), 0.5f);
    float* o = out + bi * 256 + 32 * ib;
    for (int t = 0; t < 32; ++t) {
        const int l = t >> 3, j = t & 7;
        const uint32_t seven = (sw >> (7 * l)) & 0x7Fu;
        const uint32_t neg = j < 7 ? (seven >> j) & 1u : (__popc(seven) & 1u);
        // page 4 halves the grid bytes (doubled units); page 3 uses them as they are
        const float mag = __fmul_rn(static_cast<float>(grid[4 * blk[F::kIdxOff + 8 * ib + (t >> 2)] + (t & 3)]),
                                    F::kGridScale);
        o[t] = __fmul_rn(neg ? -mag : mag, db);
    }
}

int launch_dequant_q4k(const uint8_t* W, float* out, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nblocks = N * (K / 256);
    const int64_t threads = nblocks * 4;
    qg_dequant_q4k_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(W, out, nblocks);
    return launch_status();
}

int launch_dequant_iq3(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nblocks = N * (K / 256);
    const int64_t threads = nblocks * 8;
    qg_dequant_iq3_kernel<FmtIQ3T><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(W, grid, out, nblocks);
    return launch_status();
}

int launch_dequant_iq3xxs(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nblocks = N * (K / 256);
    const int64_t threads = nblocks * 8;
    qg_dequant_iq3_kernel<FmtIQ3XXST><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(W, grid, out,
                                                                                              nblocks);
    return launch_status();
}

}  // namespace qg
