// Fused-dequantisation GEMV over block-quantised weights, fp32 FMA path.
//
//   Y[m][n] = sum_k w[n][k] * X[m][k],   m < MT <= 4 tokens per launch
//
// w is never materialised: it is decoded in registers from the block bytes
// and dotted with x.  Formats:
//   Q4_K  page 1 "Rewriting picoLM in Python", dequantize_q4_K
//   IQ3   page 4 "iq3_pack.py" (fmt=5), module docstring and decode, and
//         page 3's IQ3_XXS byte order of the same fields
//
// CTA = RG row groups x 8 consumer warps + 1 producer warp (FmtQ4KT2: 16
// consumer warps, two per column); a tile is RG*32 consecutive rows, walked
// in units of 8 super-block columns.
//   * The producer warp posts, per unit, one 2D tensor-map TMA
//     (cp.async.bulk.tensor) per super-block column, a [tile rows][box] box
//     of that column's blocks, plus the x slice of each token (Q4_K: one bulk
//     copy per token, contiguous; IQ3: one tensor-map box per token in a
//     padded layout), all completing on the stage's `full` mbarrier.  It
//     reuses a stage once every consumer warp has arrived on its `empty`
//     mbarrier: no CTA-wide barrier in the steady state.  With the
//     weight-prefetch flag the weights of the first stages are posted before
//     the programmatic-dependent-launch wait, x after it.
//   * Consumer warp (rg, c) takes block column c.  Lane L decodes two rows,
//     L&15 and (L&15)+16 of its row group, half L>>4 of each block (128
//     weights), so every x load serves two rows; the halves of a row meet in
//     one shuffle when the tile ends.  FmtQ4KT2 gives each half of a column
//     its own warp (lane L: sub-block pair L>>4 of the warp's half).  Box rows of 144 B (Q4_K) or 112 B
//     (IQ3) are odd multiples of 16 bytes, so eight lanes loading eight rows
//     with 16-byte loads hit eight distinct bank groups.
//   * Per-row partial sums stay in registers across a tile's units and are
//     reduced over the 8 column warps through a double-buffered smem array
//     once per tile (one named barrier among the consumers), or across a
//     cluster's CTAs through DSMEM when the tile's K is split over a cluster.
//
// Q4_K arithmetic, sub-block j (a = d*sc_j, b = dmin*mn_j, c the integer in
// [0, 15] nearest b/a; see q4k_offset):
//   sum_l (a*q_l - b) * x_l = a * sum_l (q_l - c) * x_l - (b - a*c) * sum_l x_l
// sum_l x_l is computed once per (column, token) by the warp, shared by its
// 32 rows; q_l - c is formed exactly while each nibble is an fp32 subnormal
// against x pre-scaled by powers of two.  IQ3: one byte permute per weight
// joins a grid byte (from a lane-replicated table of zero-interleaved grid
// rows) and a sign byte (from a table of the 128 sign fields) into the fp32
// subnormal +-g * 2^-149; the sub-block factor d*(0.5+code) is applied per
// sub-block.  Slices of x outside the directly handled range are rescaled
// by a power of two (see q4k_stage_x and iq3_stage_x).
#pragma once
#include <cuda_fp16.h>

#include "common.cuh"

namespace qg {

constexpr int kRows = 32;        // rows per row group (one per lane)
constexpr int kCols = 8;         // super-block columns per unit (one per consumer warp)
constexpr int kMaxStages = 6;
constexpr int kSmemPerSM = 233472;   // 228 KB per SM on sm_103
constexpr int kSmemPerCTA = 232448;  // 227 KB max dynamic smem per CTA
constexpr int kSmemReserve = 1024;   // per-CTA system reservation

// x of one super-block column and token in a ring stage: two halves of 128
// floats, half 1 starting F::kXH floats after half 0.  IQ3 pads (kXH =
// kXHalf = 132): the 4-float gap puts the halves 16 bytes apart modulo the
// 128-byte bank period, so the lanes of a two-row decode (lanes 0-15 on
// half 0, 16-31 on half 1, reading the same offset in their half) load x
// without a bank conflict.  Q4_K stages x contiguously (kXH = 128): there
// the conflict costs less than the padded copy.
constexpr int kXHalf = 132;
constexpr int kXCol = 2 * kXHalf;  // padded floats per column and token (1056 bytes)

// Stage layouts.  Row-copy formats: one bulk copy per row chunk, each row in
// its own slot (kRowStride apart).  FmtQ4KT: one 2D tensor-map TMA per
// super-block column, landing as [tile rows][144 B] boxes (a unit is kCols
// boxes); 144 B = 9 x 16 B, so eight lanes reading eight consecutive rows
// with 16-byte loads hit eight distinct bank groups.
// kCols of a format: super-block columns per unit = consumer warps per row
// group.
// Tensor-map formats load box kBoxBytes wide starting at the block's byte
// offset rounded down to 16: Q4_K blocks (144 B = 9 x 16) start aligned; an
// IQ3 block (98 B) starts 0..14 bytes into its 112-byte box.  112 B = 7 x 16
// is also an odd multiple of 16, so rows stay conflict-free.
struct FmtQ4K {
    static constexpr int kBytes = 144;
    static constexpr int kCols = qg::kCols;
    static constexpr int kRowStride = kCols * 144 + 16;  // 1168 = 73 * 16 (odd)
    static constexpr int kWPC = 1;                         // consumer warps per column
    static constexpr bool kIQ3 = false;
    static constexpr bool kTMA = false;
    static constexpr int kBoxBytes = 0;
    static constexpr int kXH = 128;
};
template <int C>
struct FmtQ4KTc {
    static constexpr int kBytes = 144;
    static constexpr int kCols = C;
    static constexpr int kRowStride = C * 144;  // bytes per tile row per unit (C boxes of 144 B)
    static constexpr int kWPC = 1;              // consumer warps per column
    static constexpr bool kIQ3 = false;
    static constexpr bool kTMA = true;
    static constexpr int kBoxBytes = 144;
    static constexpr int kXH = 128;  // x staged contiguously (one bulk copy per token)
};
using FmtQ4KT = FmtQ4KTc<kCols>;
// The same stage layout with two consumer warps per column, one per half of
// each block (lane L: rows L&15 and (L&15)+16, sub-block pair L>>4 of the
// warp's half): 16 warps per unit, for launches that leave SMs with at most
// one tile.  The SM's issue rate still bounds a unit's decode; the gain is in
// the prologue work of the fused kernels, which the 16 warps share.
struct FmtQ4KT2 : FmtQ4KTc<kCols> {
    static constexpr int kWPC = 2;
};
// IQ3 block layouts (98 bytes, same fields, two orders):
//   FmtIQ3T    page 4 "iq3_pack.py": 64 index bytes @0, eight u32 @64, fp16 d
//              @96; value = d*(0.5+code)*0.5 * grid*0.5 * sign
//   FmtIQ3XXST page 3 (llama.cpp IQ3_XXS): fp16 d @0, 64 index bytes @2,
//              eight u32 @66; value = d*(0.5+s)*0.5 * grid * sign
// kDbScale folds the constant factors into the sub-block factor
// d*(0.5+code)*kDbScale that multiplies the raw grid bytes.
struct FmtIQ3T {
    static constexpr int kBytes = 98;
    static constexpr int kCols = qg::kCols;
    static constexpr int kRowStride = kCols * 112;  // bytes per tile row per unit (kCols boxes of 112 B)
    static constexpr int kWPC = 1;                  // consumer warps per column
    static constexpr bool kIQ3 = true;
    static constexpr bool kTMA = true;
    static constexpr int kBoxBytes = 112;
    static constexpr int kXH = kXHalf;  // x staged in the padded layout (one 2D box per token)
    static constexpr int kIdxOff = 0, kWordOff = 64, kDOff = 96;
    static constexpr float kDbScale = 0.25f;
    static constexpr float kGridScale = 0.5f;  // the magnitude of a grid byte
};
struct FmtIQ3XXST : FmtIQ3T {
    static constexpr int kIdxOff = 2, kWordOff = 66, kDOff = 0;
    static constexpr float kDbScale = 0.5f;
    static constexpr float kGridScale = 1.f;
};

// IQ3 tables in smem, shared by all consumer warps.
// Grid: lane-replicated so every gather is conflict-free: for grid row i,
// lane L reads the 8 bytes at 256*i + 8*L, the row's four bytes laid out as
// [g0, 0, g1, 0] [g2, 0, g3, 0].  Signs: for each 7-bit sign field s7 two
// words of sign bytes, [s0 s1 s2 s3] [s4 s5 s6 s7] with s_k = 0x80 when
// weight k is negative (the eighth sign: the parity of the seven, page 4
// decode).  One byte permute of a grid word and a sign word then gives an
// fp32 with the sign of weight k at bit 31 and its grid byte at bits 0-7:
// the exact value +-g * 2^-149, which q4k-style pre-scaled x (2^88) turns
// into a normal product.  Replicated per half-warp lane: lane L reads the 8
// bytes at 128*s7 + 8*(L & 15).
constexpr int kIQ3GridBytes = 256 * 32 * 8;
constexpr int kIQ3SignBytes = 128 * 16 * 8;
constexpr int kIQ3TableBytes = kIQ3GridBytes + kIQ3SignBytes;


__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Split-K over a thread-block cluster: up to kMaxCluster CTAs share a tile,
// one K chunk each, and meet in the first CTA's shared memory.
constexpr int kMaxCluster = 8;
__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

struct Layout {
    int full, empty, sx, red, cred, ss, table, stage0, stage_bytes, xoff, aoff, total;
};

// Fused prologue / epilogue of a GEMV (page 2 "Candle", RmsNorm::forward
// and Block::forward: h = rmsnorm(x) before q/k/v and gate/up,
// down(silu(gate) * up), residual adds).  Kernel template FUSE selects the
// prologue: 0 none, kFuseNorm x' = x * g / rms(x), kFuseSwiGLU
// x' = silu(x) * up.  R[i] (residual of matrix i, [M][N[i]], may be Y[i]
// itself) is added to the output when not null, with any FUSE.
constexpr int kFuseNorm = 1;
constexpr int kFuseSwiGLU = 2;
struct Fuse {
    const float* g;    // RMSNorm weight [K]
    const float* up;   // SwiGLU up operand [M][K]
    const float* R[4]; // residuals (one per matrix of the group), or null
    float eps;         // RMSNorm epsilon
};

// Up to kMaxGroup matrices that share X and K, processed by one launch.
// Tiles are numbered across the group: matrix i owns tiles
// [tile0[i], tile0[i+1]).
constexpr int kMaxGroup = 4;
struct Group {
    const uint8_t* W[kMaxGroup];
    float* Y[kMaxGroup];
    int64_t N[kMaxGroup];
    int64_t tile0[kMaxGroup + 1];
    int count;
};

// Tensor maps of the group's matrices: bytes [N][K/256*B], box kBoxBytes x
// tile rows; and of X viewed as [M*K/128][128] fp32 with 132 x 16 boxes
// (one box = the padded x of one unit's 8 columns for one token).
struct TMaps {
    CUtensorMap m[kMaxGroup];
    CUtensorMap xm;
};
constexpr uint32_t kXBoxBytes = 16 * kXHalf * 4;  // 8448

// Matrix that owns global tile `tile`.
__device__ __forceinline__ int group_find(const Group& G, int64_t tile) {
    int i = 0;
#pragma unroll
    for (int k = 1; k < kMaxGroup; ++k)
        if (k < G.count && tile >= G.tile0[k]) i = k;
    return i;
}

// Dynamic smem layout of qg_gemv_kernel<F, MT, RG> with `stages` stages;
// xh = F::kXH when x is staged with the weights, 0 when it is read from
// global memory.
__host__ __device__ inline Layout make_layout(bool iq3, int MT, int xh, int RG, int stages, int row_stride,
                                              int cols = kCols, int fuse = 0, int wpc = 1) {
    Layout L;
    const int warps = RG * cols * wpc;
    L.full = 0;
    L.empty = 8 * kMaxStages;
    L.sx = 128;
    L.red = L.sx + align_up(warps * MT * 8 * 4, 128);
    L.cred = L.red + align_up(2 * warps * MT * kRows * 4, 128);
    L.ss = L.cred + align_up(kMaxCluster * MT * (RG * kRows + 1) * 4, 128);
    L.table = L.ss + align_up(2 * warps * MT * 4, 128);
    L.stage0 = L.table + (iq3 ? kIQ3TableBytes : 0);
    L.xoff = align_up(RG * kRows * row_stride, 128);
    L.aoff = L.xoff + MT * cols * 8 * xh;  // xh: F::kXH with x staged, else 0
    // prologue operands staged beside x: RMSNorm weight (shared by the
    // tokens) or the SwiGLU up operand (per token), 1 KB per column
    L.stage_bytes = L.aoff + (fuse == kFuseNorm ? cols * 1024 : fuse == kFuseSwiGLU ? MT * cols * 1024 : 0);
    L.total = L.stage0 + stages * L.stage_bytes;
    return L;
}

// ------------------------------------------------------------ Q4_K helpers
// The 12 packed bytes (little-endian words P0, P1, P2) -> eight 6-bit scales
// and mins, four per result word (byte k of sc03 = sc[k], of sc47 = sc[4+k]).
// Page 1: j < 4 -> low six bits of byte j (scale) / j+4 (min); j >= 4 ->
// low (scale) / high (min) nibble of byte j+4, with bits 6-7 of byte j-4
// (scale) / byte j (min) as bits 4-5.
__device__ __forceinline__ void q4k_scale_min_words(uint32_t P0, uint32_t P1, uint32_t P2, uint32_t& sc03,
                                                    uint32_t& mn03, uint32_t& sc47, uint32_t& mn47) {
    sc03 = P0 & 0x3F3F3F3Fu;
    mn03 = P1 & 0x3F3F3F3Fu;
    sc47 = (P2 & 0x0F0F0F0Fu) | ((P0 >> 2) & 0x30303030u);
    mn47 = ((P2 >> 4) & 0x0F0F0F0Fu) | ((P1 >> 2) & 0x30303030u);
}

__device__ __forceinline__ float byte_f(uint32_t w, int k) { return static_cast<float>((w >> (8 * k)) & 0xFFu); }
__device__ __forceinline__ float half_lo(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
}

// SiLU (page 2 "Candle", Block::forward's silu): z * sigmoid(z).
// exp and the division by the fast hardware paths (__expf, __fdividef:
// relative errors of a few ulp, far inside the GEMV's 1e-5 tolerance); for
// z << 0 the denominator passes 2^126 or overflows and __fdividef gives 0,
// the limit (the true value is below 1e-36 in size there).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// Range of the staged x slices that q4k_half2 takes as they are: the
// largest |x| of a token's 256-value slice in [2^-24, 2^39).  Products of a
// nibble (at most 15) with x are then normal fp32 numbers after the 2^76..2^88
// pre-scaling below, and no pre-scaled value overflows.  A slice outside
// that range (but finite) is first multiplied by 2^-e, e the exponent of its
// largest |x| clamped to [-100, 100], and the column's partial sums by 2^e
// afterwards: every finite x is handled, only the cost differs.
constexpr uint32_t kXExpLo = 127 - 24, kXExpHi = 127 + 39;  // biased exponents

// Per-warp x preparation for one Q4_K super-block column (256 x values per
// token; half 1, x[128..255], starts XH floats after half 0):
// sx[m*8 + j] = sum of x over sub-block j (the dmin*mn term's factor), and
// the x values (in smem) are scaled in place by 2^(88-c), c = 4*(high
// nibble) + 8*(odd byte), the bit offsets at which q4k_half2 finds each
// nibble.  A token whose slice lies outside the range above is also scaled
// by 2^-e first (sx too); e2[m] = 2^e then (1 otherwise), and the return
// value, the same in every lane, says whether any token was.  With FUSE the
// prologue (kFuseNorm: x * g, sum of x^2 into ss; kFuseSwiGLU: silu(x) * up)
// is applied first, reading g or up at ab (+ m * astride), laid out like x;
// the range test, sx and the scaling see the result.  Callers must fence
// the written x against the next bulk copy into the same slot.
template <int MT, int XH, int FUSE = 0>
__device__ __forceinline__ bool q4k_stage_x(float* xb, int64_t xstride, const float* ab, int64_t astride, float* sx,
                                            float (&ss)[MT], float (&e2)[MT], int M, int lane) {
    bool rescaled = false;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        e2[m] = 1.f;
        if (MT == 1 || m < M) {
            const int off = (lane >> 4) * XH + ((lane >> 2) & 3) * 32 + (lane & 3) * 8;
            float* xp = xb + m * xstride + off;
            float4 a = *reinterpret_cast<const float4*>(xp);
            float4 b = *reinterpret_cast<const float4*>(xp + 4);
            if constexpr (FUSE == kFuseNorm) {
                // RMSNorm prologue: sum of squares of the raw x (1/rms is
                // applied to the finished row sums), then x * g
                ss[m] = fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(a.z, a.z, fmaf(a.w, a.w, ss[m]))));
                ss[m] = fmaf(b.x, b.x, fmaf(b.y, b.y, fmaf(b.z, b.z, fmaf(b.w, b.w, ss[m]))));
                const float4 ga = *reinterpret_cast<const float4*>(ab + off);
                const float4 gb = *reinterpret_cast<const float4*>(ab + off + 4);
                a = make_float4(a.x * ga.x, a.y * ga.y, a.z * ga.z, a.w * ga.w);
                b = make_float4(b.x * gb.x, b.y * gb.y, b.z * gb.z, b.w * gb.w);
            } else if constexpr (FUSE == kFuseSwiGLU) {
                // SwiGLU prologue: silu(gate) * up, gate being x
                const float4 ua = *reinterpret_cast<const float4*>(ab + m * astride + off);
                const float4 ub = *reinterpret_cast<const float4*>(ab + m * astride + off + 4);
                a = make_float4(silu(a.x) * ua.x, silu(a.y) * ua.y, silu(a.z) * ua.z, silu(a.w) * ua.w);
                b = make_float4(silu(b.x) * ub.x, silu(b.y) * ub.y, silu(b.z) * ub.z, silu(b.w) * ub.w);
            }
            // largest |x| of the slice (fmaxf passes over NaN; an all-NaN lane
            // reads as the largest value and takes the rescaled path, whose
            // result is NaN as it must be)
            const float mx = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                                   fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
            const uint32_t top = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
            const uint32_t be = top >> 23;
            if (top != 0u && (be < kXExpLo || be >= kXExpHi)) {  // the same in every lane
                const int e = min(max(static_cast<int>(be) - 127, -100), 100);
                const float s = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
                a = make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
                b = make_float4(b.x * s, b.y * s, b.z * s, b.w * s);
                e2[m] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
                rescaled = true;
            }
            float sm = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
            sm += __shfl_xor_sync(0xffffffffu, sm, 1);
            sm += __shfl_xor_sync(0xffffffffu, sm, 2);
            if ((lane & 3) == 0) sx[m * 8 + (lane >> 2)] = sm;
            const float se = ((lane >> 2) & 1) ? 0x1p84f : 0x1p88f;  // even byte
            const float so = se * 0x1p-8f;                           // odd byte
            a = make_float4(a.x * se, a.y * so, a.z * se, a.w * so);
            b = make_float4(b.x * se, b.y * so, b.z * se, b.w * so);
            *reinterpret_cast<float4*>(xp) = a;
            *reinterpret_cast<float4*>(xp + 4) = b;
        }
    }
    return rescaled;
}

// q4k_stage_x for one half of a column, when two warps share the column
// (FmtQ4KT2): xh = the half's 128 x values of token 0 (token m at
// xh + m*xstride), ah likewise for the prologue operand; lane L takes
// x[32*(L>>3) + 4*(L&7) .. +3], sub-block 4h + (L>>3), and writes its sum to
// sx[m*8 + 4h + (L>>3)].  The range test covers the half's 128 values.
template <int MT, int FUSE = 0>
__device__ __forceinline__ bool q4k_stage_x_half(float* xh, int64_t xstride, const float* ah, int64_t astride,
                                                 float* sx, int h, float (&ss)[MT], float (&e2)[MT], int M,
                                                 int lane) {
    bool rescaled = false;
    const int off = (lane >> 3) * 32 + (lane & 7) * 4;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        e2[m] = 1.f;
        if (MT == 1 || m < M) {
            float* xp = xh + m * xstride + off;
            float4 a = *reinterpret_cast<const float4*>(xp);
            if constexpr (FUSE == kFuseNorm) {
                ss[m] = fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(a.z, a.z, fmaf(a.w, a.w, ss[m]))));
                const float4 ga = *reinterpret_cast<const float4*>(ah + off);
                a = make_float4(a.x * ga.x, a.y * ga.y, a.z * ga.z, a.w * ga.w);
            } else if constexpr (FUSE == kFuseSwiGLU) {
                const float4 ua = *reinterpret_cast<const float4*>(ah + m * astride + off);
                a = make_float4(silu(a.x) * ua.x, silu(a.y) * ua.y, silu(a.z) * ua.z, silu(a.w) * ua.w);
            }
            const float mx = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w)));
            const uint32_t top = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
            const uint32_t be = top >> 23;
            if (top != 0u && (be < kXExpLo || be >= kXExpHi)) {  // the same in every lane
                const int e = min(max(static_cast<int>(be) - 127, -100), 100);
                const float sc = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
                a = make_float4(a.x * sc, a.y * sc, a.z * sc, a.w * sc);
                e2[m] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
                rescaled = true;
            }
            float sm = (a.x + a.y) + (a.z + a.w);
            sm += __shfl_xor_sync(0xffffffffu, sm, 1);
            sm += __shfl_xor_sync(0xffffffffu, sm, 2);
            sm += __shfl_xor_sync(0xffffffffu, sm, 4);
            if ((lane & 7) == 0) sx[m * 8 + 4 * h + (lane >> 3)] = sm;
            const float se = ((lane >> 3) & 1) ? 0x1p84f : 0x1p88f;  // even byte of the sub-block's nibbles
            const float so = se * 0x1p-8f;                           // odd byte
            *reinterpret_cast<float4*>(xp) = make_float4(a.x * se, a.y * so, a.z * se, a.w * so);
        }
    }
    return rescaled;
}

// Offset of a Q4_K sub-block with scale a = d*sc and min b = dmin*mn: the
// integer c in [0, 15] nearest b/a.  For any integer c
//   sum_l (a*q_l - b)*x_l = a * sum_l (q_l - c)*x_l - (b - a*c) * sum_l x_l,
// and with the nearest one every term on the right is at most twice the
// |w*x| of its weight (|b - a*c| <= a/2, and |a*(q - c)| <= 2|a*q - b| for
// q != c), so the factored sum keeps the accuracy of the per-weight one even
// where d*sc*q and dmin*mn cancel.  b - a*c is exact in fp32 whenever c > 0
// (both products are exact and their exponents are close).  a = 0 gives an
// infinite or NaN quotient: fmaxf drops the NaN and the clamp takes the rest.
__device__ __forceinline__ float q4k_offset(float a, float b) {
    return fminf(fmaxf(rintf(__fdividef(b, a)), 0.f), 15.f);
}

// Half of one Q4_K super-block column for two rows (x pre-scaled by
// q4k_stage_x; half 1 of x XH floats after half 0).  Lane L of a warp takes
// rows L&15 and (L&15)+16 of the tile and half h = L>>4 of the block
// (sub-blocks 4h..4h+3, weights 128h..128h+127), so every x load serves two
// rows; the two halves of a row meet with one shuffle at the end of the
// tile.  blk: the row-(L&15) block in smem; rstride: bytes from a row to the
// row 16 below.  Per sub-block the offset c above is taken off every nibble
// while it is still an fp32 subnormal (q*2^-149 - c*2^-149 is exact), the
// min term is (b - a*c) * sum(x), then the scaled sum of (q - c)*x.  With
// RESCALE the column's sums are formed apart and multiplied by e2[m] (the
// 2^e of a token whose slice q4k_stage_x rescaled) before they join acc.
//
// NG = 2 takes both sub-block pairs of the half (g = 0, 1); NG = 1 only the
// pair g = g1 (sub-blocks 4h+2g1 and 4h+2g1+1), for kernels whose two lanes
// L and L^16 split a half between them (FmtQ4KT2).
template <int MT, int XH, bool RESCALE, int NG = 2>
__device__ __forceinline__ void q4k_half2(const uint8_t* blk, int rstride, int h, const float* xb, int64_t xstride,
                                          const float* sx, int M, const float (&e2)[MT], float (&acc)[2][MT],
                                          int g1 = 0) {
    if constexpr (RESCALE && MT > 1) {
        // the rare rescaled column: one token at a time, which needs far fewer
        // registers than the MT-token decode and its separate column sums
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                float a1[2][1] = {{acc[0][m]}, {acc[1][m]}};
                const float e1[1] = {e2[m]};
                q4k_half2<1, XH, true, NG>(blk, rstride, h, xb + m * xstride, xstride, sx + m * 8, 1, e1, a1, g1);
                acc[0][m] = a1[0][0];
                acc[1][m] = a1[1][0];
            }
        }
        return;
    }
    float dd[2], dm[2];
    uint32_t scw[2], mnw[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint4 hd = *reinterpret_cast<const uint4*>(blk + j * rstride);
        dd[j] = h2f(hd.x);
        dm[j] = h2f(hd.x >> 16);
        // scales / mins of sub-blocks 4h..4h+3 (page 1 packing: j >= 4 straddles)
        scw[j] = h ? ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u)) : (hd.y & 0x3F3F3F3Fu);
        mnw[j] = h ? (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u)) : (hd.z & 0x3F3F3F3Fu);
    }
    float part[2][MT];
    float (&tgt)[2][MT] = RESCALE ? part : acc;
    if constexpr (RESCALE) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) part[j][m] = 0.f;
    }
    const uint8_t* qb = blk + 16 + 64 * h;
    const float* xq = xb + XH * h;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        const int g = NG == 2 ? gi : g1;
        // sub-blocks 4h+2g (low nibbles) and 4h+2g+1 (high nibbles) of each row
        float al61[2], ah61[2];  // a * 2^61 (the pre-scaling of x is 2^-61 in the products)
        f2 ol[2], oh[2];         // -c at the subnormal scales of the nibbles' bit offsets
        // the two rows' scale arithmetic as packed pairs (row 0, row 1)
        const f2 dd2{dd[0], dd[1]}, dm2{dm[0], dm[1]};
        const f2 a0 = fmul2(dd2, f2{byte_f(scw[0], 2 * g), byte_f(scw[1], 2 * g)});
        const f2 a1 = fmul2(dd2, f2{byte_f(scw[0], 2 * g + 1), byte_f(scw[1], 2 * g + 1)});
        const f2 b0 = fmul2(dm2, f2{byte_f(mnw[0], 2 * g), byte_f(mnw[1], 2 * g)});
        const f2 b1 = fmul2(dm2, f2{byte_f(mnw[0], 2 * g + 1), byte_f(mnw[1], 2 * g + 1)});
        const f2 c0{q4k_offset(a0.x, b0.x), q4k_offset(a0.y, b0.y)};
        const f2 c1{q4k_offset(a1.x, b1.x), q4k_offset(a1.y, b1.y)};
        f2 r0 = b0, r1 = b1;  // b - a*c, exact where it matters
        ffma2(r0, f2{-a0.x, -a0.y}, c0);
        ffma2(r1, f2{-a1.x, -a1.y}, c1);
        const f2 al2 = fmul2(a0, f2{0x1p61f, 0x1p61f}), ah2 = fmul2(a1, f2{0x1p61f, 0x1p61f});
        al61[0] = al2.x;
        al61[1] = al2.y;
        ah61[0] = ah2.x;
        ah61[1] = ah2.y;
        ol[0] = fmul2(f2{c0.x, c0.x}, f2{-0x1p-149f, -0x1p-141f});
        ol[1] = fmul2(f2{c0.y, c0.y}, f2{-0x1p-149f, -0x1p-141f});
        oh[0] = fmul2(f2{c1.x, c1.x}, f2{-0x1p-145f, -0x1p-137f});
        oh[1] = fmul2(f2{c1.y, c1.y}, f2{-0x1p-145f, -0x1p-137f});
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (MT == 1 || m < M) {
                const float s0 = sx[m * 8 + 4 * h + 2 * g], s1 = sx[m * 8 + 4 * h + 2 * g + 1];
                tgt[0][m] = fmaf(-r0.x, s0, tgt[0][m]);
                tgt[0][m] = fmaf(-r1.x, s1, tgt[0][m]);
                tgt[1][m] = fmaf(-r0.y, s0, tgt[1][m]);
                tgt[1][m] = fmaf(-r1.y, s1, tgt[1][m]);
            }
        }
        f2 al[2][MT], ah[2][MT];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) al[j][m] = ah[j][m] = f2{0.f, 0.f};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint4 q[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) q[j] = *reinterpret_cast<const uint4*>(qb + j * rstride + 32 * g + 16 * hh);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kl = 64 * g + 16 * hh + 4 * e;  // weights kl..kl+3 (low nibbles), +32 (high)
                float4 xl[MT], xh[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (MT == 1 || m < M) {
                        xl[m] = *reinterpret_cast<const float4*>(xq + m * xstride + kl);
                        xh[m] = *reinterpret_cast<const float4*>(xq + m * xstride + kl + 32);
                    }
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t v = e == 0 ? q[j].x : e == 1 ? q[j].y : e == 2 ? q[j].z : q[j].w;
                    const uint32_t u = v >> 16;
                    // each nibble in place as an fp32 subnormal, then q - c
                    f2 l01{__uint_as_float(v & 0xFu), __uint_as_float(v & 0xF00u)};
                    f2 l23{__uint_as_float(u & 0xFu), __uint_as_float(u & 0xF00u)};
                    f2 h01{__uint_as_float(v & 0xF0u), __uint_as_float(v & 0xF000u)};
                    f2 h23{__uint_as_float(u & 0xF0u), __uint_as_float(u & 0xF000u)};
                    fadd2(l01, ol[j]);
                    fadd2(l23, ol[j]);
                    fadd2(h01, oh[j]);
                    fadd2(h23, oh[j]);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (MT == 1 || m < M) {
                            ffma2(al[j][m], l01, f2{xl[m].x, xl[m].y});
                            ffma2(al[j][m], l23, f2{xl[m].z, xl[m].w});
                            ffma2(ah[j][m], h01, f2{xh[m].x, xh[m].y});
                            ffma2(ah[j][m], h23, f2{xh[m].z, xh[m].w});
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (MT == 1 || m < M) {
                    tgt[j][m] = fmaf(al61[j], al[j][m].x + al[j][m].y, tgt[j][m]);
                    tgt[j][m] = fmaf(ah61[j], ah[j][m].x + ah[j][m].y, tgt[j][m]);
                }
            }
        }
    }
    if constexpr (RESCALE) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (MT == 1 || m < M) acc[j][m] = fmaf(part[j][m], e2[m], acc[j][m]);
    }
}

// Sign words (S0, S1) of the sign field at bits 7l..7l+6 of sw (see
// kIQ3SignBytes); lane_s = 8 * (lane & 15).
__device__ __forceinline__ uint2 iq3_signs(const uint8_t* sg, uint32_t sw, int l, uint32_t lane_s) {
    const uint32_t off = (l == 0 ? (sw << 7) : (sw >> (7 * l - 7))) & 0x3F80u;
    return *reinterpret_cast<const uint2*>(sg + (off | lane_s));
}

// Grid row of the index byte `byte` of word w: 8 bytes [g0,0,g1,0][g2,0,g3,0].
__device__ __forceinline__ uint2 iq3_grid(const uint8_t* tb, uint32_t w, int byte, uint32_t lane8) {
    const uint32_t off = prmt(w, lane8, 4u | (static_cast<uint32_t>(byte) << 4) | (5u << 8) | (5u << 12));
    return *reinterpret_cast<const uint2*>(tb + off);
}

// Signed grid value as an fp32 subnormal: byte P of grid word g (P = 0 or 2;
// bytes 1 and 3 of g are zero) at bits 0-7, sign byte K of s at bits 24-31.
template <int P, int K>
__device__ __forceinline__ float iq3_val(uint32_t g, uint32_t s) {
    return __uint_as_float(prmt(g, s, static_cast<uint32_t>(P) | (1u << 4) | (1u << 8) | ((4u + K) << 12)));
}

// Half h of the IQ3 super-block of column COL from its 112-byte TMA box row
// (the block starts (98*COL) mod 16 bytes in): vi = index bytes 32h..32h+31,
// vs = sign/scale words 4h..4h+3, dbits = the fp16 d (field offsets of F).
template <class F, int COL>
__device__ __forceinline__ void iq3_load_half(const uint8_t* boxrow, int h, uint32_t (&vi)[8], uint32_t (&vs)[4],
                                              uint32_t& dbits) {
    constexpr int OFF = (COL * 98) & 15;
    constexpr int OI = OFF + F::kIdxOff, W0 = OI >> 2, SH = 8 * (OI & 3);          // index bytes
    constexpr int OW = OFF + F::kWordOff - 64, W0w = OW >> 2, SHw = 8 * (OW & 3);  // sign/scale words
    constexpr int OD = OFF + F::kDOff;                                             // d
    uint32_t w[12];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const uint4 t = *reinterpret_cast<const uint4*>(boxrow + 32 * h + 16 * i);
        w[4 * i] = t.x; w[4 * i + 1] = t.y; w[4 * i + 2] = t.z; w[4 * i + 3] = t.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) vi[i] = SH ? __funnelshift_r(w[W0 + i], w[W0 + i + 1], SH) : w[W0 + i];
    uint32_t u[8];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint4 t = *reinterpret_cast<const uint4*>(boxrow + 64 + 16 * h + 16 * i);
        u[4 * i] = t.x; u[4 * i + 1] = t.y; u[4 * i + 2] = t.z; u[4 * i + 3] = t.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) vs[i] = SHw ? __funnelshift_r(u[W0w + i], u[W0w + i + 1], SHw) : u[W0w + i];
    dbits = *reinterpret_cast<const uint32_t*>(boxrow + (OD & ~3)) >> (8 * (OD & 3));
}

// Two rows (r, r+16), half h of an IQ3 super-block each, against MT tokens:
// the layout of q4k_half2 (one x load serves both rows).  xq = x of the
// block + 128h, pre-scaled by 2^88 (iq3_stage_x).  Each weight is one byte
// permute (iq3_val: grid byte and sign as an fp32 subnormal) and half a
// packed FMA; the sub-block factor d*(0.5+code)*kDbScale*2^61 undoes the
// scaling.  With RESCALE the column's sums are formed apart and multiplied
// by e2[m] (a token whose slice iq3_stage_x rescaled) before they join acc.
template <int MT, class F, bool RESCALE>
__device__ __forceinline__ void iq3_half2(const uint32_t (&vi)[2][8], const uint32_t (&vs)[2][4], const uint32_t (&dbits)[2],
                                          const uint8_t* tb, const uint8_t* sg, uint32_t lane8, uint32_t lane_s,
                                          const float* xq, int64_t xstride, int M, const float (&e2)[MT],
                                          float (&acc)[2][MT]) {
    if constexpr (RESCALE && MT > 1) {
        // the rare rescaled column: one token at a time (fewer registers)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                float a1[2][1] = {{acc[0][m]}, {acc[1][m]}};
                const float e1[1] = {e2[m]};
                iq3_half2<1, F, true>(vi, vs, dbits, tb, sg, lane8, lane_s, xq + m * xstride, xstride, 1, e1, a1);
                acc[0][m] = a1[0][0];
                acc[1][m] = a1[1][0];
            }
        }
        return;
    }
    float part[2][MT];
    float (&tgt)[2][MT] = RESCALE ? part : acc;
    if constexpr (RESCALE) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) part[r][m] = 0.f;
    }
    // sub-block factor d*(0.5+code)*kDbScale*2^61 = fma(1 + code/16, 16 d', -15.5 d')
    // with d' = d*kDbScale*2^61: 1 + code/16 is the float with the code as
    // the top four mantissa bits; every term is exact, so is the result
    float d16[2], d155[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float d = h2f(dbits[r]);
        d16[r] = d * (16.f * F::kDbScale * 0x1p61f);
        d155[r] = d * (15.5f * F::kDbScale * 0x1p61f);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f2 dot[2][MT];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) dot[r][m] = f2{0.f, 0.f};
#pragma unroll
        for (int l = 0; l < 4; ++l) {
            uint2 T[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) T[r] = iq3_signs(sg, vs[r][j], l, lane_s);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int PI = 8 * j + 2 * l + hf;  // index byte within the half
                float4 x[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (MT == 1 || m < M) x[m] = *reinterpret_cast<const float4*>(xq + m * xstride + 32 * j + 8 * l + 4 * hf);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint2 g = iq3_grid(tb, vi[r][PI >> 2], PI & 3, lane8);
                    const uint32_t t = hf ? T[r].y : T[r].x;  // signs of weights 4hf..4hf+3 of the field
                    const f2 w01{iq3_val<0, 0>(g.x, t), iq3_val<2, 1>(g.x, t)};
                    const f2 w23{iq3_val<0, 2>(g.y, t), iq3_val<2, 3>(g.y, t)};
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (MT == 1 || m < M) {
                            ffma2(dot[r][m], w01, f2{x[m].x, x[m].y});
                            ffma2(dot[r][m], w23, f2{x[m].z, x[m].w});
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float f = __uint_as_float(((vs[r][j] >> 9) & 0x00780000u) | 0x3F800000u);
            const float db = fmaf(f, d16[r], -d155[r]);
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (MT == 1 || m < M) tgt[r][m] = fmaf(db, dot[r][m].x + dot[r][m].y, tgt[r][m]);
        }
    }
    if constexpr (RESCALE) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (MT == 1 || m < M) acc[r][m] = fmaf(part[r][m], e2[m], acc[r][m]);
    }
}

// Per-warp x preparation for one IQ3 column (the warp's own copy, 256
// values per token, halves XH floats apart): every value scaled in place by
// 2^88, so that a grid byte held as an fp32 subnormal (g * 2^-149) times x
// is a normal number.  A token whose largest |x| lies outside [2^-24, 2^39)
// (the range of q4k_stage_x) is first scaled by 2^-e as well, e the exponent
// of its largest |x| clamped to [-100, 100]; e2[m] = 2^e then (1 otherwise),
// and the return value, the same in every lane, says whether any token was.
// Callers must fence the written x against the next copy into the slot.
template <int MT, int XH>
__device__ __forceinline__ bool iq3_stage_x(float* xb, int64_t xstride, int M, int lane, float (&e2)[MT]) {
    bool rescaled = false;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        e2[m] = 1.f;
        if (MT == 1 || m < M) {
            float* xp = xb + m * xstride + (lane >> 4) * XH + (lane & 15) * 8;
            float4 a = *reinterpret_cast<const float4*>(xp);
            float4 b = *reinterpret_cast<const float4*>(xp + 4);
            const float mx = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                                   fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
            const uint32_t top = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
            const uint32_t be = top >> 23;
            if (top != 0u && (be < kXExpLo || be >= kXExpHi)) {  // the same in every lane
                const int e = min(max(static_cast<int>(be) - 127, -100), 100);
                const float s = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
                a = make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
                b = make_float4(b.x * s, b.y * s, b.z * s, b.w * s);
                e2[m] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
                rescaled = true;
            }
            constexpr float k88 = 0x1p88f;
            *reinterpret_cast<float4*>(xp) = make_float4(a.x * k88, a.y * k88, a.z * k88, a.w * k88);
            *reinterpret_cast<float4*>(xp + 4) = make_float4(b.x * k88, b.y * k88, b.z * k88, b.w * k88);
        }
    }
    return rescaled;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Launch flag: W and the grid are not written by the preceding kernel in the
// stream, so they may be prefetched before the grid dependency is resolved.
constexpr int kFlagPrefetchWeights = 1;
// Launch flag bits 8-11: cluster size C > 1 (split-K over a cluster of C CTAs
// per tile; the grid is ntiles * C, CTA rank r takes chunk r).
constexpr int kFlagClusterShift = 8;

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Store v at the same shared-memory offset as p in cluster CTA `rank`.
__device__ __forceinline__ void st_cluster_f32(const void* p, uint32_t rank, float v) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void named_barrier_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(N) : "memory");
}
__device__ __forceinline__ void named_barrier_sync_n(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ------------------------------------------------------------ the kernel
// Threads: RG*8 consumer warps, then one producer warp.
// x is staged in shared memory with each unit (Q4_K contiguous, IQ3 in the
// padded layout above) and decoded two rows per lane (lane L: rows L&15 and
// (L&15)+16, half L>>4 of each block).
template <class F, int MT, int RG, int MINB, int FUSE = 0>
__global__ void __launch_bounds__(RG * F::kCols * F::kWPC * 32 + 32, MINB)
    qg_gemv_kernel(const __grid_constant__ Group G, const __grid_constant__ TMaps T, const __grid_constant__ Fuse Fz,
                const uint8_t* __restrict__ grid, const float* __restrict__ X, int M, int64_t K, int stages,
                unsigned* status, int flags) {
    constexpr int kRGWarps = F::kCols * F::kWPC;   // consumer warps per row group
    constexpr int kWarps = RG * kRGWarps;          // consumer warps
    constexpr int kConsumerThreads = kWarps * 32;
    constexpr int kTileRows = RG * kRows;
    extern __shared__ __align__(128) uint8_t smem[];
    const int nb = static_cast<int>(K / 256);
    const int nchunks = (nb + F::kCols - 1) / F::kCols;
    const int64_t ntiles = G.tile0[G.count];
    constexpr int XH = F::kXH;  // floats from half 0 to half 1 of a staged x column
    const Layout L = make_layout(F::kIQ3, MT, XH, RG, stages, F::kRowStride, F::kCols, FUSE, F::kWPC);
    static_assert(FUSE == 0 || !F::kIQ3, "fused prologues run on the Q4_K path");
    static_assert(F::kWPC == 1 || (F::kWPC == 2 && !F::kIQ3 && RG == 1), "two warps per column: Q4_K, one row group");
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    float* sxw = reinterpret_cast<float*>(smem + L.sx);
    float* red = reinterpret_cast<float*>(smem + L.red);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    static_assert(F::kTMA, "weights arrive through the format's tensor map");
    static_assert(F::kCols == 8, "one x box holds 8 columns");
    static_assert(F::kIQ3 || RG == 1, "in-place x scaling needs one warp per column");

    // Programmatic dependent launch: let the next kernel in the stream get
    // scheduled now.  Without the weight-prefetch flag, wait for the previous
    // kernel before touching any global memory; with it, only W and the grid
    // (weights, never written by the previous kernel) are read before the wait.
    grid_launch_dependents();
    const bool prefetch = (flags & kFlagPrefetchWeights) != 0;
    if (!prefetch) grid_dependency_wait();
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        fence_mbar_init();
    }
    // IQ3 tables (lane-replicated grid and sign bytes), built by threads
    // tid, tid + nt, ...  With several tokens the consumer warps build them
    // while the producer's first copies are in flight (3 % faster at four
    // tokens); the one-token kernel measured 1.5-3 % faster building them
    // with every thread before the producer starts.
    constexpr bool kTablesInConsumers = F::kIQ3 && MT > 1;
    auto build_tables = [&](int tid, int nt) {
        // grid rows as bytes [g0, 0, g1, 0] [g2, 0, g3, 0], 32 lane copies
        uint32_t* tbl = reinterpret_cast<uint32_t*>(smem + L.table);
        for (int i = tid; i < 256 * 32; i += nt) {
            const uint32_t g = *reinterpret_cast<const uint32_t*>(grid + 4 * (i >> 5));
            tbl[2 * i] = (g & 0xFFu) | ((g & 0xFF00u) << 8);
            tbl[2 * i + 1] = ((g >> 16) & 0xFFu) | ((g >> 8) & 0xFF0000u);
        }
        // sign bytes: s8 = the seven stored signs + their parity (page 4,
        // decode); word h holds weights 4h..4h+3, 0x80 in byte k if negative
        uint32_t* sgt = reinterpret_cast<uint32_t*>(smem + L.table + kIQ3GridBytes);
        for (int i = tid; i < 128 * 32; i += nt) {
            const uint32_t s7 = static_cast<uint32_t>(i) >> 5;  // 32 words per field: 16 copies of (S0, S1)
            const uint32_t s8 = s7 | ((__popc(s7) & 1u) << 7);
            const uint32_t nib = (s8 >> (4 * (i & 1))) & 15u;
            sgt[i] = ((nib & 1u) << 7) | ((nib & 2u) << 14) | ((nib & 4u) << 21) | ((nib & 8u) << 28);
        }
    };
    if constexpr (F::kIQ3 && !kTablesInConsumers) build_tables(threadIdx.x, blockDim.x);
    __syncthreads();  // the barriers are initialised (and the one-token tables built)

    // Cluster split-K: this CTA takes chunk `crank` of tile blockIdx.x / csize.
    const int csize = (flags >> kFlagClusterShift) & 15;
    const bool clus = csize > 1;
    const int crank = clus ? static_cast<int>(cluster_ctarank()) : 0;
    const int64_t tile_first = clus ? blockIdx.x / csize : blockIdx.x;
    if (clus) cluster_arrive_relaxed();  // phase 0: every CTA of the cluster has started
    const int64_t my_tiles =
        clus ? (tile_first < ntiles ? 1 : 0)
             : (static_cast<int64_t>(blockIdx.x) < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0);
    const int64_t U = clus ? my_tiles : my_tiles * nchunks;

    if (warp == kWarps) {
        // ---------------- producer warp
        // Unit bookkeeping is incremental (stage, chunk, tile): no division
        // in the loop.
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        // bring the tensor-map descriptors in before the first copies (the x
        // map's first use sits on the dependency chain)
        if (lane < G.count) prefetch_tensormap(&T.m[lane]);
        if (XH == kXHalf && lane == 31) prefetch_tensormap(&T.xm);
        struct Pos {
            int s, c;
            int64_t tile, row0;
            int gi, rows;
        };
        auto first_pos = [&]() {
            Pos p{0, crank, tile_first, 0, 0, 0};
            p.gi = group_find(G, p.tile);
            p.row0 = (p.tile - G.tile0[p.gi]) * kTileRows;
            p.rows = static_cast<int>(min64(kTileRows, G.N[p.gi] - p.row0));
            return p;
        };
        auto next_pos = [&](Pos& p) {
            if (++p.s == stages) p.s = 0;
            if (++p.c == nchunks) {
                p.c = 0;
                p.tile += gridDim.x;
                if (p.tile < ntiles) {
                    p.gi = group_find(G, p.tile);
                    p.row0 = (p.tile - G.tile0[p.gi]) * kTileRows;
                    p.rows = static_cast<int>(min64(kTileRows, G.N[p.gi] - p.row0));
                }
            }
        };
        auto post = [&](const Pos& p, bool do_w, bool do_x, bool expect) {
            const int kc = min(F::kCols, nb - p.c * F::kCols);
            uint8_t* st = smem + L.stage0 + p.s * L.stage_bytes;
            // kc boxes of kBoxBytes x kTileRows; rows past N (and bytes past
            // the row end) arrive as zeros and count in full toward the
            // transaction bytes.
            constexpr uint32_t kBox = kTileRows * F::kBoxBytes;
            // x, padded layout: one 132 x 16 box per token (the unit's 8
            // columns as 16 padded halves; halves past the chunk are never
            // read); contiguous layout: one bulk copy per token
            constexpr bool kXBox = (XH == kXHalf);
            constexpr int kAuxTokens = FUSE == kFuseSwiGLU ? 1 : 0;  // up: per token; g: once
            if (expect) {
                const uint32_t aux = FUSE == 0 ? 0u : (kAuxTokens ? M : 1) * kc * 1024;
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[p.s],
                                          kc * kBox + M * (kXBox ? kXBoxBytes : kc * 1024) + aux);
                __syncwarp();
            }
            if (do_w && lane == 0)
                for (int b = 0; b < kc; ++b)
                    tma_load_2d(st + b * kBox, &T.m[p.gi], ((p.c * F::kCols + b) * F::kBytes) & ~15,
                                static_cast<int>(p.row0), &full[p.s], pol_w);
            if (do_x && lane < M) {
                if constexpr (kXBox)
                    tma_load_2d(st + L.xoff + lane * kXBoxBytes, &T.xm, 0,
                                static_cast<int>((lane * K) / 128 + p.c * (2 * F::kCols)), &full[p.s], pol_x);
                else
                    bulk_g2s(st + L.xoff + lane * F::kCols * 1024,
                             X + lane * K + static_cast<int64_t>(p.c) * F::kCols * 256, kc * 1024, &full[p.s], pol_x);
            }
            // prologue operand slices, laid out like x: the RMSNorm weight is
            // a model weight (it streams with W, before the dependency wait);
            // the SwiGLU up operand belongs to the dependency chain, as x does
            if constexpr (FUSE == kFuseNorm) {
                if (do_w && lane == 0)
                    bulk_g2s(st + L.aoff, Fz.g + static_cast<int64_t>(p.c) * F::kCols * 256, kc * 1024, &full[p.s],
                             pol_x);
            } else if constexpr (FUSE == kFuseSwiGLU) {
                if (do_x && lane < M)
                    bulk_g2s(st + L.aoff + lane * F::kCols * 1024,
                             Fz.up + lane * K + static_cast<int64_t>(p.c) * F::kCols * 256, kc * 1024, &full[p.s],
                             pol_x);
            }
        };
        Pos p = first_pos();
        int64_t u0 = 0;
        if (prefetch) {
            // weights of the first stages stream while the previous kernel runs
            const int64_t pre = min64(stages, U);
            Pos q = p;
            for (int64_t u = 0; u < pre; ++u, next_pos(q)) post(q, true, false, true);
            grid_dependency_wait();
            for (int64_t u = 0; u < pre; ++u, next_pos(p)) post(p, false, true, false);
            u0 = pre;
        }
        uint32_t round = 0;  // completed passes over the ring before unit u
        for (int64_t u = 0; u < u0; ++u)
            if (static_cast<int>(u % stages) == stages - 1) ++round;
        for (int64_t u = u0; u < U; ++u, next_pos(p)) {
            if (u >= stages) mbar_wait_bounded(&empty[p.s], (round - 1) & 1u, status);
            post(p, true, true, true);
            if (p.s == stages - 1) ++round;
        }
        if (clus) {  // the producer takes part in both cluster barrier phases
            __syncwarp();
            cluster_wait();
            cluster_arrive_release();
            cluster_wait();
        }
        return;
    }

    // ---------------- consumer warps
    if constexpr (kTablesInConsumers) {
        build_tables(threadIdx.x, kConsumerThreads);  // the producer never reads them
        named_barrier_sync<kConsumerThreads>(1);
    }
    if (prefetch) grid_dependency_wait();  // x and Y belong to the dependency chain
    const int rg = warp / kRGWarps, cw = warp % F::kCols;
    const int hw = (warp / F::kCols) % F::kWPC;  // FmtQ4KT2: the warp's half of its column
    // two rows per lane (acc2[j]: row (lane&15) + 16j, half lane>>4)
    float acc2[2][MT];
    float ss[MT];  // RMSNorm prologue: this lane's part of sum(x^2) over the tile's units
#pragma unroll
    for (int m = 0; m < MT; ++m) acc2[0][m] = acc2[1][m] = ss[m] = 0.f;
    const uint32_t lane8 = static_cast<uint32_t>(lane) * 8u, lane_s = static_cast<uint32_t>(lane & 15) * 8u;
    int64_t tile_count = 0;

    int s = 0, c = crank;
    uint32_t phase = 0;
    int64_t tile = tile_first;
    int gi = 0;
    int64_t row0 = 0, Ni = 0;
    int rows = 0;
    auto load_tile = [&]() {
        gi = group_find(G, tile);
        row0 = (tile - G.tile0[gi]) * kTileRows;
        Ni = G.N[gi];
        rows = static_cast<int>(min64(kTileRows, Ni - row0));
    };
    if (U > 0) load_tile();
    // Residual epilogue of the prologue kernels (FUSE != 0): the thread that
    // finishes (token m, row rr) of a tile (thread m * 32 + rr of the tile's
    // finishing CTA) loads its residual when the tile starts, so the load's
    // latency hides behind the decode.  The FUSE = 0 kernels, which also run
    // the plain GEMV, read it in the epilogue: the extra live register costs
    // the large one-token GEMV 1.5-2 % and spills in the two-token kernel.
    static_assert(MT * kTileRows <= kConsumerThreads, "one finishing thread per output");
    float rpre = 0.f;
    for (int64_t u = 0; u < U; ++u) {
        const int kc = min(F::kCols, nb - c * F::kCols);
        const uint8_t* st = smem + L.stage0 + s * L.stage_bytes;
        if (FUSE != 0 && c == crank && Fz.R[gi] && crank == 0 && threadIdx.x < MT * kTileRows) {
            const int m = threadIdx.x / kTileRows, rr = threadIdx.x % kTileRows;
            if ((MT == 1 || m < M) && rr < rows) rpre = Fz.R[gi][m * Ni + row0 + rr];
        }
        mbar_wait_bounded(&full[s], phase, status);

        if (cw < kc) {
            const float* xb = reinterpret_cast<const float*>(st + L.xoff) + cw * 2 * XH;
            const int64_t xstride = F::kCols * 2 * XH;
            if constexpr (!F::kIQ3 && F::kWPC == 2) {
                // half hw of the column: its x (128 values per token), then
                // sub-block pair lane>>4 of the half for rows lane&15 and +16
                float* sxp = sxw + warp * MT * 8;
                const float* ab = reinterpret_cast<const float*>(st + L.aoff) + cw * 256 + hw * 128;
                float e2[MT];
                const bool rescaled = q4k_stage_x_half<MT, FUSE>(const_cast<float*>(xb) + hw * XH, xstride, ab,
                                                                 F::kCols * 256, sxp, hw, ss, e2, M, lane);
                __syncwarp();
                const uint8_t* blk = st + cw * (kTileRows * F::kBytes) + (lane & 15) * F::kBytes;
                if (rescaled)  // x outside the direct range (rare; the same in every lane)
                    q4k_half2<MT, XH, true, 1>(blk, 16 * F::kBytes, hw, xb, xstride, sxp, M, e2, acc2, lane >> 4);
                else
                    q4k_half2<MT, XH, false, 1>(blk, 16 * F::kBytes, hw, xb, xstride, sxp, M, e2, acc2, lane >> 4);
                fence_proxy_async_smem();  // x was written: order it before the slot's next copy
            } else if constexpr (!F::kIQ3) {
                float* sxp = sxw + warp * MT * 8;
                const float* ab = reinterpret_cast<const float*>(st + L.aoff) + cw * 256;
                float e2[MT];
                const bool rescaled =
                    q4k_stage_x<MT, XH, FUSE>(const_cast<float*>(xb), xstride, ab, F::kCols * 256, sxp, ss, e2, M, lane);
                __syncwarp();
                const uint8_t* blk = st + cw * (kTileRows * F::kBytes) + (lane & 15) * F::kBytes;
                if (rescaled)  // x outside the direct range (rare; the same in every lane)
                    q4k_half2<MT, XH, true>(blk, 16 * F::kBytes, lane >> 4, xb, xstride, sxp, M, e2, acc2);
                else
                    q4k_half2<MT, XH, false>(blk, 16 * F::kBytes, lane >> 4, xb, xstride, sxp, M, e2, acc2);
                fence_proxy_async_smem();  // x was written: order it before the slot's next copy
            } else {
                // two rows per lane, half a block each (TMA layout): rows
                // rg*32 + (lane&15) and +16, half lane>>4
                const int hl = lane >> 4;
                const uint8_t* box = st + cw * (kTileRows * F::kBoxBytes) + (rg * kRows + (lane & 15)) * F::kBoxBytes;
                uint32_t vi[2][8], vs[2][4], dbits[2];
                switch (cw) {
#define QG_IQ3_HALF(C)                                                          \
    case C:                                                                     \
        iq3_load_half<F, C>(box, hl, vi[0], vs[0], dbits[0]);                      \
        iq3_load_half<F, C>(box + 16 * F::kBoxBytes, hl, vi[1], vs[1], dbits[1]);  \
        break;
                    QG_IQ3_HALF(0) QG_IQ3_HALF(1) QG_IQ3_HALF(2) QG_IQ3_HALF(3)
                    QG_IQ3_HALF(4) QG_IQ3_HALF(5) QG_IQ3_HALF(6)
                    default:
                        iq3_load_half<F, 7>(box, hl, vi[0], vs[0], dbits[0]);
                        iq3_load_half<F, 7>(box + 16 * F::kBoxBytes, hl, vi[1], vs[1], dbits[1]);
                        break;
#undef QG_IQ3_HALF
                }
                const uint8_t* tb = smem + L.table;
                float e2[MT];
                bool rescaled;
                if constexpr (RG == 1) {
                    rescaled = iq3_stage_x<MT, XH>(const_cast<float*>(xb), xstride, M, lane, e2);
                    __syncwarp();
                } else {
                    // the column's x is shared by its RG warps: row group 0
                    // scales it and publishes the rescale factors (slots
                    // alternate with the unit, so a slot is rewritten only
                    // after both warps passed the next unit's barrier), then
                    // the column's warps meet on a named barrier
                    float* ef = reinterpret_cast<float*>(smem + L.ss) + ((u & 1) * F::kCols + cw) * MT;
                    if (rg == 0) {
                        rescaled = iq3_stage_x<MT, XH>(const_cast<float*>(xb), xstride, M, lane, e2);
                        if (lane == 0)
#pragma unroll
                            for (int m = 0; m < MT; ++m) ef[m] = e2[m];  // the same in every lane
                    }
                    named_barrier_sync_n(2 + cw, RG * 32);
                    if (rg != 0) {
                        rescaled = false;
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            e2[m] = ef[m];
                            rescaled |= e2[m] != 1.f;
                        }
                    }
                }
                const uint8_t* sg = tb + kIQ3GridBytes;
                const float* xq = xb + XH * hl;
                if (rescaled)  // rare; the same in every lane
                    iq3_half2<MT, F, true>(vi, vs, dbits, tb, sg, lane8, lane_s, xq, xstride, M, e2, acc2);
                else
                    iq3_half2<MT, F, false>(vi, vs, dbits, tb, sg, lane8, lane_s, xq, xstride, M, e2, acc2);
                fence_proxy_async_smem();  // x was written: order it before the slot's next copy
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        if (clus || c == nchunks - 1) {
            // reduce the 8 column warps' partial sums of each row, write Y
            float* rb = red + (tile_count & 1) * (kWarps * MT * kRows);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                // lanes L and L^16 hold the two halves (FmtQ4KT2: the two
                // sub-block pairs of the warp's half) of rows L&15 and (L&15)+16
                const float s0 = acc2[0][m] + __shfl_xor_sync(0xffffffffu, acc2[0][m], 16);
                const float s1 = acc2[1][m] + __shfl_xor_sync(0xffffffffu, acc2[1][m], 16);
                rb[(warp * MT + m) * kRows + lane] = lane < 16 ? s0 : s1;
                acc2[0][m] = acc2[1][m] = 0.f;
            }
            // RMSNorm prologue: each warp's sum of x^2 (its columns, all of
            // the tile's chunks) per token
            float* ssw = reinterpret_cast<float*>(smem + L.ss) + (tile_count & 1) * (kWarps * MT);
            if constexpr (FUSE == kFuseNorm) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float t = ss[m];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                    if (lane == 0) ssw[warp * MT + m] = t;
                    ss[m] = 0.f;
                }
            }
            named_barrier_sync<kConsumerThreads>(1);
            // finished row sum -> output: times 1/rms(x) of the token, plus the residual
            auto finish = [&](int m, int rr, float sum, float sumsq) {
                if constexpr (FUSE == kFuseNorm) sum *= rsqrtf(sumsq / static_cast<float>(K) + Fz.eps);
                const int64_t o = m * Ni + row0 + rr;
                if (Fz.R[gi]) sum += FUSE != 0 ? rpre : Fz.R[gi][o];  // prologue kernels: loaded at the tile's start
                G.Y[gi][o] = sum;
            };
            if (clus) {
                // this chunk's row sums (and sum of x^2) -> slot crank of the
                // first CTA; after the cluster barrier it adds the slots in
                // rank order (deterministic)
                float* cred = reinterpret_cast<float*>(smem + L.cred);
                float* cssq = cred + kMaxCluster * MT * kTileRows;
                __syncwarp();
                cluster_wait();  // phase 0: all CTAs of the cluster are running
                for (int t = threadIdx.x; t < MT * kTileRows; t += kConsumerThreads) {
                    const int m = t / kTileRows, rr = t % kTileRows;
                    const int g = rr / kRows, ln = rr % kRows;
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < kRGWarps; ++w) sum += rb[((g * kRGWarps + w) * MT + m) * kRows + ln];
                    st_cluster_f32(cred + crank * MT * kTileRows + t, 0, sum);
                }
                if (FUSE == kFuseNorm && threadIdx.x < MT) {
                    float q = 0.f;
                    for (int w = 0; w < kWarps; ++w) q += ssw[w * MT + threadIdx.x];
                    st_cluster_f32(cssq + crank * MT + threadIdx.x, 0, q);
                }
                __syncwarp();
                cluster_arrive_release();
                cluster_wait();
                if (crank == 0) {
                    for (int t = threadIdx.x; t < MT * kTileRows; t += kConsumerThreads) {
                        const int m = t / kTileRows, rr = t % kTileRows;
                        if ((MT == 1 || m < M) && rr < rows) {
                            float sum = 0.f, sq = 0.f;
                            for (int q = 0; q < csize; ++q) sum += cred[q * MT * kTileRows + t];
                            if (FUSE == kFuseNorm)
                                for (int q = 0; q < csize; ++q) sq += cssq[q * MT + m];
                            finish(m, rr, sum, sq);
                        }
                    }
                }
            } else {
                for (int t = threadIdx.x; t < MT * kTileRows; t += kConsumerThreads) {
                    const int m = t / kTileRows, rr = t % kTileRows;
                    const int g = rr / kRows, ln = rr % kRows;
                    if ((MT == 1 || m < M) && rr < rows) {
                        float sum = 0.f, sq = 0.f;
#pragma unroll
                        for (int w = 0; w < kRGWarps; ++w) sum += rb[((g * kRGWarps + w) * MT + m) * kRows + ln];
                        if (FUSE == kFuseNorm)
                            for (int w = 0; w < kWarps; ++w) sq += ssw[w * MT + m];
                        finish(m, rr, sum, sq);
                    }
                }
            }
            ++tile_count;
        }
        // advance (stage ring, chunk, tile) without division
        if (++s == stages) {
            s = 0;
            phase ^= 1u;
        }
        if (++c == nchunks) {
            c = 0;
            tile += gridDim.x;
            if (tile < ntiles) load_tile();
        }
    }
    if (clus && U == 0) {  // no unit (never with grid = ntiles * C): still pass both phases
        cluster_wait();
        cluster_arrive_release();
        cluster_wait();
    }
}

}  // namespace qg
