// Fused-dequantisation GEMV over block-quantised weights, fp32 FMA path.
//
//   Y[m][n] = sum_k w[n][k] * X[m][k],   m < M <= 32
//
// w is never materialised: each thread decodes one 256-weight super-block
// in registers and dots it with x.  Formats:
//   Q4_K  page 1 "Rewriting picoLM in Python", dequantize_q4_K
//   IQ3   page 4 "iq3_pack.py" (fmt=5), module docstring and decode
//
// Work decomposition (one CTA per SM, persistent over row tiles):
//   * a tile is kRows=32 consecutive rows; the CTA walks the tile's K range in
//     chunks of kCols=8 super-block columns;
//   * per chunk, warp 0 issues one cp.async.bulk per row (the row's 8 blocks
//     are contiguous in HBM) into a padded smem slot, plus one bulk copy per
//     token of the matching x slice; completion is tracked by an mbarrier;
//   * lane r of warp c decodes block (row r, column c): the 8 lanes of a
//     quarter-warp read 8 different rows (conflict-free thanks to the odd
//     multiple-of-16 row stride) and all 32 lanes read the same x (broadcast);
//   * per-row partial sums stay in registers across chunks and are reduced
//     over the 8 warps through smem once per tile.
//
// Q4_K arithmetic: for sub-block j, sum_l (d*sc_j*q_l - dmin*mn_j)*x_l =
// (d*sc_j) * sum_l q_l*x_l - (dmin*mn_j) * sum_l x_l; sum_l x_l is computed
// once per (block column, token) by the warp and shared by all 32 rows.
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace qg {

constexpr int kRows = 32;
constexpr int kCols = 8;
constexpr int kThreads = kRows * kCols;  // 256: 8 warps
constexpr int kMaxStages = 6;
constexpr int kSmemLimit = 232448;       // 227 KB dynamic smem per CTA on sm_103

struct FmtQ4K {
    static constexpr int kBytes = 144;
    static constexpr int kRowStride = kCols * 144 + 16;  // 1168 = 73 * 16
    static constexpr bool kIQ3 = false;
};
struct FmtIQ3 {
    static constexpr int kBytes = 98;
    static constexpr int kRowStride = kCols * 98;        // 784 = 49 * 16
    static constexpr bool kIQ3 = true;
};

// IQ3 grid table in smem, lane-replicated so every gather is conflict-free:
// for grid row i, lane L reads word 64*i + L (halves of magnitudes 0,1) and
// word 64*i + 32 + L (halves of magnitudes 2,3).  64 KB.
constexpr int kIQ3TableBytes = 256 * 64 * 4;

struct Layout {
    int bars, sx, red, table, stage0, stage_bytes, xoff, total;
};

__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }
__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__host__ __device__ inline Layout make_layout(bool iq3, int MT, bool xs, int stages, int row_stride) {
    Layout L;
    L.bars = 0;
    L.sx = 128;
    L.red = L.sx + align_up(kCols * MT * 8 * 4, 128);
    L.table = L.red + align_up(kCols * MT * kRows * 4, 128);
    L.stage0 = L.table + (iq3 ? kIQ3TableBytes : 0);
    L.xoff = align_up(kRows * row_stride, 128);
    L.stage_bytes = L.xoff + (xs ? MT * kCols * 1024 : 0);
    L.total = L.stage0 + stages * L.stage_bytes;
    return L;
}

// ------------------------------------------------------------ Q4_K helpers
// The 12 packed bytes (three little-endian words P0, P1, P2) -> eight 6-bit
// scales and mins, four per word, byte k of the result word = field 4*h + k.
// Page 1: j < 4 -> low six bits of byte j / j+4; j >= 4 -> low/high nibble of
// byte j+4 plus bits 6-7 of byte j-4 / byte j as bits 4-5.
__device__ __forceinline__ void q4k_scale_min_words(uint32_t P0, uint32_t P1, uint32_t P2, uint32_t& sc03,
                                                    uint32_t& mn03, uint32_t& sc47, uint32_t& mn47) {
    sc03 = P0 & 0x3F3F3F3Fu;
    mn03 = P1 & 0x3F3F3F3Fu;
    sc47 = (P2 & 0x0F0F0F0Fu) | ((P0 >> 2) & 0x30303030u);
    mn47 = ((P2 >> 4) & 0x0F0F0F0Fu) | ((P1 >> 2) & 0x30303030u);
}

__device__ __forceinline__ float byte_f(uint32_t w, int k) { return static_cast<float>((w >> (8 * k)) & 0xFFu); }

__device__ __forceinline__ float half_lo(uint32_t h) { return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu))); }
__device__ __forceinline__ float half_hi(uint32_t h) { return __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16))); }

// One Q4_K super-block (144 bytes at blk, smem) against MT tokens of x.
// sx[m*8 + j] = sum of x over sub-block j for token m.
// Nibbles become exact fp32 through the fp16 magic 0x6400|q (= 1024 + q):
// low nibbles give 1024+q, high nibbles (left in place) 1024+16q, and the
// mixed f16->f32 add of -1024 yields q or 16q exactly; the 1/16 is folded
// into the sub-block scale (exact, a power of two).
template <int MT>
__device__ __forceinline__ void q4k_block(const uint8_t* blk, const float* xb, int64_t xstride, const float* sx,
                                          int M, float (&acc)[MT]) {
    const uint4 h = *reinterpret_cast<const uint4*>(blk);
    const float d = h2f(h.x), dmin = h2f(h.x >> 16);
    uint32_t sc03, mn03, sc47, mn47;
    q4k_scale_min_words(h.y, h.z, h.w, sc03, mn03, sc47, mn47);
    float mt[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) mt[m] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float dmn = dmin * byte_f(j < 4 ? mn03 : mn47, j & 3);
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (m < M) mt[m] = fmaf(dmn, sx[m * 8 + j], mt[m]);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t scw = g < 2 ? sc03 : sc47;
        const float dl = d * byte_f(scw, (2 * g) & 3);
        const float dh = d * byte_f(scw, (2 * g + 1) & 3) * 0.0625f;
        f2 al[MT], ah[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) al[m] = ah[m] = f2{0.f, 0.f};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint4 q = *reinterpret_cast<const uint4*>(blk + 16 + 32 * g + 16 * hh);
            const uint32_t qv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t v = qv[e], v8 = v >> 8;
                const uint32_t A = (v & 0x000F000Fu) | 0x64006400u;   // bytes 0,2 low nibbles
                const uint32_t C = (v8 & 0x000F000Fu) | 0x64006400u;  // bytes 1,3 low nibbles
                const uint32_t B = (v & 0x00F000F0u) | 0x64006400u;   // bytes 0,2 high nibbles (x16)
                const uint32_t D = (v8 & 0x00F000F0u) | 0x64006400u;  // bytes 1,3 high nibbles (x16)
                const f2 l01{add_f16_f32(A, -1024.f), add_f16_f32(C, -1024.f)};
                const f2 l23{add_f16hi_f32(A, -1024.f), add_f16hi_f32(C, -1024.f)};
                const f2 h01{add_f16_f32(B, -1024.f), add_f16_f32(D, -1024.f)};
                const f2 h23{add_f16hi_f32(B, -1024.f), add_f16hi_f32(D, -1024.f)};
                const int kl = 64 * g + 16 * hh + 4 * e;  // weights kl..kl+3 (low), +32 (high)
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < M) {
                        const float4 xl = *reinterpret_cast<const float4*>(xb + m * xstride + kl);
                        const float4 xh = *reinterpret_cast<const float4*>(xb + m * xstride + kl + 32);
                        ffma2(al[m], l01, f2{xl.x, xl.y});
                        ffma2(al[m], l23, f2{xl.z, xl.w});
                        ffma2(ah[m], h01, f2{xh.x, xh.y});
                        ffma2(ah[m], h23, f2{xh.z, xh.w});
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                acc[m] = fmaf(dl, al[m].x + al[m].y, acc[m]);
                acc[m] = fmaf(dh, ah[m].x + ah[m].y, acc[m]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] -= mt[m];
}

// One IQ3 super-block against MT tokens.  rowp is the 16-byte aligned start
// of the row's 8-block chunk in smem; the block sits at byte COL*98, so its
// alignment (and every field offset below) is a compile-time constant.
// Each 4-weight group gathers its grid row from the lane-replicated fp16
// table (exact magnitudes), flips signs in the fp16 domain (sign bits moved
// to bits 15/31 by one multiply, no carries between the shifted copies),
// converts to fp32 and FMAs.  The sub-block factor d*(0.5+code)*0.5 and the
// grid's 0.5 are applied once per 32 weights (exact: at most 16 significant
// bits).
template <int COL, int MT>
__device__ __forceinline__ void iq3_block(const uint8_t* rowp, const uint32_t* tbl, uint32_t lane4, const float* xb,
                                          int64_t xstride, int M, float (&acc)[MT]) {
    constexpr int S0 = COL * 98, A0 = S0 & ~15, OFF = S0 - A0;
    uint32_t w[28];
#pragma unroll
    for (int i = 0; i < 7; ++i) {
        const uint4 t = *reinterpret_cast<const uint4*>(rowp + A0 + 16 * i);
        w[4 * i] = t.x;
        w[4 * i + 1] = t.y;
        w[4 * i + 2] = t.z;
        w[4 * i + 3] = t.w;
    }
    constexpr int PD = OFF + 96;
    const float d = h2f(w[PD >> 2] >> (8 * (PD & 3)));
    const uint8_t* tb = reinterpret_cast<const uint8_t*>(tbl);
#pragma unroll
    for (int ib = 0; ib < 8; ++ib) {
        const int PW = OFF + 64 + 4 * ib;
        const uint32_t sw = (PW & 3) == 0 ? w[PW >> 2] : __funnelshift_r(w[PW >> 2], w[(PW >> 2) + 1], 8 * (PW & 3));
        const float db = d * (static_cast<float>(sw >> 28) + 0.5f) * 0.25f;
        f2 dot[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) dot[m] = f2{0.f, 0.f};
#pragma unroll
        for (int l = 0; l < 4; ++l) {
            const uint32_t seven = (sw >> (7 * l)) & 0x7Fu;
            const uint32_t s8 = seven | ((__popc(seven) & 1u) << 7);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int PI = OFF + 8 * ib + 2 * l + hf;  // grid index byte of weights 8l+4hf..+3
                const uint32_t off = prmt(w[PI >> 2], lane4, 4u | (static_cast<uint32_t>(PI & 3) << 4) | (5u << 8) | (5u << 12));
                const uint32_t* tp = reinterpret_cast<const uint32_t*>(tb + off);
                uint32_t h01 = tp[0], h23 = tp[32];
                const uint32_t k01 = hf ? ((1u << 11) + (1u << 26)) : ((1u << 15) + (1u << 30));
                const uint32_t k23 = hf ? ((1u << 9) + (1u << 24)) : ((1u << 13) + (1u << 28));
                h01 ^= (s8 * k01) & 0x80008000u;
                h23 ^= (s8 * k23) & 0x80008000u;
                const f2 w01{half_lo(h01), half_hi(h01)};
                const f2 w23{half_lo(h23), half_hi(h23)};
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < M) {
                        const float4 x = *reinterpret_cast<const float4*>(xb + m * xstride + 32 * ib + 8 * l + 4 * hf);
                        ffma2(dot[m], w01, f2{x.x, x.y});
                        ffma2(dot[m], w23, f2{x.z, x.w});
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (m < M) acc[m] = fmaf(db, dot[m].x + dot[m].y, acc[m]);
    }
}

// ------------------------------------------------------------ the kernel
template <class F, int MT, bool XS>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ grid, const float* __restrict__ X,
                float* __restrict__ Y, int M, int64_t N, int64_t K, int stages, unsigned* status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int nb = static_cast<int>(K / 256);
    const int nchunks = (nb + kCols - 1) / kCols;
    const int64_t ntiles = (N + kRows - 1) / kRows;
    const Layout L = make_layout(F::kIQ3, MT, XS, stages, F::kRowStride);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    float* sxw = reinterpret_cast<float*>(smem + L.sx);
    float* red = reinterpret_cast<float*>(smem + L.red);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t pitch = static_cast<int64_t>(nb) * F::kBytes;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    if constexpr (F::kIQ3) {
        // halves of the doubled-unit magnitudes (exact: bytes < 2048)
        uint32_t* tbl = reinterpret_cast<uint32_t*>(smem + L.table);
        for (int i = threadIdx.x; i < 256 * 32; i += kThreads) {
            const int row = i >> 5, ln = i & 31;
            const uint32_t g = *reinterpret_cast<const uint32_t*>(grid + 4 * row);
            const __half2 a = __floats2half2_rn(byte_f(g, 0), byte_f(g, 1));
            const __half2 b = __floats2half2_rn(byte_f(g, 2), byte_f(g, 3));
            tbl[64 * row + ln] = *reinterpret_cast<const uint32_t*>(&a);
            tbl[64 * row + 32 + ln] = *reinterpret_cast<const uint32_t*>(&b);
        }
    }
    __syncthreads();

    const int64_t my_tiles =
        static_cast<int64_t>(blockIdx.x) < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t U = my_tiles * nchunks;
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();

    // Warp 0: post the copies of unit u (tile, chunk) into stage u % stages.
    auto issue = [&](int64_t u) {
        const int c = static_cast<int>(u % nchunks);
        const int64_t tile = blockIdx.x + (u / nchunks) * gridDim.x;
        const int64_t row0 = tile * kRows;
        const int rows = static_cast<int>(min64(kRows, N - row0));
        const int kc = min(kCols, nb - c * kCols);
        const int s = static_cast<int>(u % stages);
        uint8_t* st = smem + L.stage0 + s * L.stage_bytes;
        const uint32_t bytes = rows * kc * F::kBytes + (XS ? M * kc * 1024 : 0);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
        __syncwarp();
        if (lane < rows)
            bulk_g2s(st + lane * F::kRowStride, W + (row0 + lane) * pitch + static_cast<int64_t>(c) * kCols * F::kBytes,
                     kc * F::kBytes, &full[s], pol_w);
        if (XS && lane < M)
            bulk_g2s(st + L.xoff + lane * kCols * 1024, X + lane * K + static_cast<int64_t>(c) * kCols * 256,
                     kc * 1024, &full[s], pol_x);
    };

    if (warp == 0)
        for (int64_t u = 0; u < min64(stages - 1, U); ++u) issue(u);

    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    const uint32_t lane4 = static_cast<uint32_t>(lane) * 4u;

    for (int64_t u = 0; u < U; ++u) {
        if (warp == 0 && u + stages - 1 < U) issue(u + stages - 1);
        const int s = static_cast<int>(u % stages);
        const int c = static_cast<int>(u % nchunks);
        const int64_t tile = blockIdx.x + (u / nchunks) * gridDim.x;
        const int64_t row0 = tile * kRows;
        const int rows = static_cast<int>(min64(kRows, N - row0));
        const int kc = min(kCols, nb - c * kCols);
        const uint8_t* st = smem + L.stage0 + s * L.stage_bytes;
        mbar_wait_bounded(&full[s], static_cast<uint32_t>((u / stages) & 1), status);

        if (warp < kc) {
            const int64_t b = static_cast<int64_t>(c) * kCols + warp;  // super-block column
            // x of this column: token m at xb + m * xstride (floats)
            const float* xb = XS ? reinterpret_cast<const float*>(st + L.xoff) + warp * 256 : X + b * 256;
            const int64_t xstride = XS ? kCols * 256 : K;
            if constexpr (!F::kIQ3) {
                // sum of x over each 32-weight sub-block, per token
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < M) {
                        const float* xp = xb + m * xstride + (lane >> 2) * 32 + (lane & 3) * 8;
                        const float4 a = *reinterpret_cast<const float4*>(xp);
                        const float4 bb = *reinterpret_cast<const float4*>(xp + 4);
                        float sm = ((a.x + a.y) + (a.z + a.w)) + ((bb.x + bb.y) + (bb.z + bb.w));
                        sm += __shfl_xor_sync(0xffffffffu, sm, 1);
                        sm += __shfl_xor_sync(0xffffffffu, sm, 2);
                        if ((lane & 3) == 0) sxw[(warp * MT + m) * 8 + (lane >> 2)] = sm;
                    }
                }
                __syncwarp();
                if (lane < rows) q4k_block<MT>(st + lane * F::kRowStride + warp * F::kBytes, xb, xstride,
                                               sxw + warp * MT * 8, M, acc);
            } else {
                if (lane < rows) {
                    const uint8_t* rowp = st + lane * F::kRowStride;
                    const uint32_t* tbl = reinterpret_cast<const uint32_t*>(smem + L.table);
                    switch (warp) {
                        case 0: iq3_block<0, MT>(rowp, tbl, lane4, xb, xstride, M, acc); break;
                        case 1: iq3_block<1, MT>(rowp, tbl, lane4, xb, xstride, M, acc); break;
                        case 2: iq3_block<2, MT>(rowp, tbl, lane4, xb, xstride, M, acc); break;
                        case 3: iq3_block<3, MT>(rowp, tbl, lane4, xb, xstride, M, acc); break;
                        case 4: iq3_block<4, MT>(rowp, tbl, lane4, xb, xstride, M, acc); break;
                        case 5: iq3_block<5, MT>(rowp, tbl, lane4, xb, xstride, M, acc); break;
                        case 6: iq3_block<6, MT>(rowp, tbl, lane4, xb, xstride, M, acc); break;
                        default: iq3_block<7, MT>(rowp, tbl, lane4, xb, xstride, M, acc); break;
                    }
                }
            }
        }
        if (c == nchunks - 1) {
            // reduce the 8 warps' partial sums of each row, write Y
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                red[(warp * MT + m) * kRows + lane] = acc[m];
                acc[m] = 0.f;
            }
            __syncthreads();
            for (int t = threadIdx.x; t < MT * kRows; t += kThreads) {
                const int m = t / kRows, r = t % kRows;
                if (m < M && r < rows) {
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < kCols; ++w) sum += red[(w * MT + m) * kRows + r];
                    Y[m * N + row0 + r] = sum;
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace qg

namespace qg {

// ------------------------------------------------ IQ3 rows not 16-byte aligned
// When K/256 is not a multiple of 8 the 98-byte rows do not start on 16-byte
// boundaries, which bulk copies require.  This path reads bytes straight
// from global memory: one warp per row, lanes over super-blocks, the grid
// staged in smem.  Correct for every K % 256 == 0; not tuned.
__global__ void __launch_bounds__(256)
    gemv_iq3_bytes_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ grid, const float* __restrict__ X,
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
            const float d = h2f(static_cast<uint32_t>(blk[96]) | (static_cast<uint32_t>(blk[97]) << 8));
            for (int ib = 0; ib < 8; ++ib) {
                const uint8_t* wp = blk + 64 + 4 * ib;
                const uint32_t sw = static_cast<uint32_t>(wp[0]) | (static_cast<uint32_t>(wp[1]) << 8) |
                                    (static_cast<uint32_t>(wp[2]) << 16) | (static_cast<uint32_t>(wp[3]) << 24);
                const float db = d * (static_cast<float>(sw >> 28) + 0.5f) * 0.25f;
                float dot[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) dot[m] = 0.f;
                for (int t = 0; t < 32; ++t) {
                    const int l = t >> 3, j = t & 7;
                    const uint32_t seven = (sw >> (7 * l)) & 0x7Fu;
                    const uint32_t neg = j < 7 ? (seven >> j) & 1u : (__popc(seven) & 1u);
                    const float mag = byte_f(g[blk[8 * ib + (t >> 2)]], t & 3);
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

// ------------------------------------------------ test-only dequantisation
// Bit-exact with the pages' fp32 evaluation order: the products and the
// difference are rounded separately (no FMA contraction).
__global__ void dequant_q4k_kernel(const uint8_t* __restrict__ W, float* __restrict__ out, int64_t nblocks) {
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

__global__ void dequant_iq3_kernel(const uint8_t* __restrict__ W, const uint8_t* __restrict__ grid,
                                   float* __restrict__ out, int64_t nblocks) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // (block, sub-block)
    if (i >= nblocks * 8) return;
    const int64_t bi = i >> 3;
    const int ib = static_cast<int>(i & 7);
    const uint8_t* blk = W + bi * 98;
    const float d = h2f(static_cast<uint32_t>(blk[96]) | (static_cast<uint32_t>(blk[97]) << 8));
    const uint8_t* wp = blk + 64 + 4 * ib;
    const uint32_t sw = static_cast<uint32_t>(wp[0]) | (static_cast<uint32_t>(wp[1]) << 8) |
                        (static_cast<uint32_t>(wp[2]) << 16) | (static_cast<uint32_t>(wp[3]) << 24);
    const float db = __fmul_rn(__fmul_rn(d, __fadd_rn(0.5f, static_cast<float>(sw >> 28))), 0.5f);
    float* o = out + bi * 256 + 32 * ib;
    for (int t = 0; t < 32; ++t) {
        const int l = t >> 3, j = t & 7;
        const uint32_t seven = (sw >> (7 * l)) & 0x7Fu;
        const uint32_t neg = j < 7 ? (seven >> j) & 1u : (__popc(seven) & 1u);
        const float mag = __fmul_rn(static_cast<float>(grid[4 * blk[8 * ib + (t >> 2)] + (t & 3)]), 0.5f);
        o[t] = __fmul_rn(neg ? -mag : mag, db);
    }
}

// ------------------------------------------------ host launchers
namespace {

int g_num_sms[64];

int sm_count(int dev) {
    if (dev < 0 || dev >= 64) return 0;
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

template <class F, int MT, bool XS>
int launch_t(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
             cudaStream_t s, unsigned* status, int dev) {
    static bool attr_done[64];
    const Layout L1 = make_layout(F::kIQ3, MT, XS, 1, F::kRowStride);
    const int stages = std::min(kMaxStages, (kSmemLimit - L1.stage0) / L1.stage_bytes);
    if (stages < 2) return QG_EINVAL;
    const Layout L = make_layout(F::kIQ3, MT, XS, stages, F::kRowStride);
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(gemv_kernel<F, MT, XS>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) !=
            cudaSuccess)
            return QG_ECUDA;
        attr_done[dev] = true;
    }
    const int64_t ntiles = (N + kRows - 1) / kRows;
    const int sms = sm_count(dev);
    if (sms <= 0) return QG_ECUDA;
    const int grid_x = static_cast<int>(min64(ntiles, sms));
    gemv_kernel<F, MT, XS><<<grid_x, kThreads, L.total, s>>>(W, grid, X, Y, M, N, K, stages, status);
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    return dev;
}

}  // namespace

// M is split into groups of at most 8 tokens; each group streams W once.
int launch_gemv_q4k(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t s,
                    unsigned* status) {
    const int dev = current_device();
    if (dev < 0) return QG_ECUDA;
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mg = std::min(8, M - m0);
        const float* Xg = X + static_cast<int64_t>(m0) * K;
        float* Yg = Y + static_cast<int64_t>(m0) * N;
        int rc;
        if (mg == 1) rc = launch_t<FmtQ4K, 1, true>(W, nullptr, Xg, Yg, mg, N, K, s, status, dev);
        else if (mg == 2) rc = launch_t<FmtQ4K, 2, true>(W, nullptr, Xg, Yg, mg, N, K, s, status, dev);
        else if (mg <= 4) rc = launch_t<FmtQ4K, 4, true>(W, nullptr, Xg, Yg, mg, N, K, s, status, dev);
        else rc = launch_t<FmtQ4K, 8, false>(W, nullptr, Xg, Yg, mg, N, K, s, status, dev);
        if (rc != QG_OK) return rc;
    }
    return QG_OK;
}

int launch_gemv_iq3(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                    cudaStream_t s, unsigned* status) {
    const int dev = current_device();
    if (dev < 0) return QG_ECUDA;
    const bool aligned = (K / 256) % 8 == 0;
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mg = std::min(8, M - m0);
        const float* Xg = X + static_cast<int64_t>(m0) * K;
        float* Yg = Y + static_cast<int64_t>(m0) * N;
        int rc;
        if (!aligned) {
            const int sms = sm_count(dev);
            if (sms <= 0) return QG_ECUDA;
            const int64_t blocks = min64((N + 7) / 8, static_cast<int64_t>(sms) * 8);
            gemv_iq3_bytes_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(W, grid, Xg, Yg, mg, N, K);
            rc = cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
        } else if (mg == 1) rc = launch_t<FmtIQ3, 1, true>(W, grid, Xg, Yg, mg, N, K, s, status, dev);
        else if (mg == 2) rc = launch_t<FmtIQ3, 2, true>(W, grid, Xg, Yg, mg, N, K, s, status, dev);
        else if (mg <= 4) rc = launch_t<FmtIQ3, 4, false>(W, grid, Xg, Yg, mg, N, K, s, status, dev);
        else rc = launch_t<FmtIQ3, 8, false>(W, grid, Xg, Yg, mg, N, K, s, status, dev);
        if (rc != QG_OK) return rc;
    }
    return QG_OK;
}

int launch_dequant_q4k(const uint8_t* W, float* out, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nblocks = N * (K / 256);
    const int64_t threads = nblocks * 4;
    dequant_q4k_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(W, out, nblocks);
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

int launch_dequant_iq3(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nblocks = N * (K / 256);
    const int64_t threads = nblocks * 8;
    dequant_iq3_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(W, grid, out, nblocks);
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

}  // namespace qg
