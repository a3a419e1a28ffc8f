// GEMV (fp32 FMA) over page 3's other codebook formats: IQ4_NL, IQ4_XS,
// IQ3_S, IQ2_XXS (llama.cpp's codebook formats as trainable students: the
// format table, get_s, eff_np and encode).  weight = eff * v, v = codebook
// entry * sign; every value is exact in fp32.
//
// Two kernels, one lane per row (32-row tiles):
//   * qg_gemv_cb_tma_kernel, every format whose rows are a multiple of 16
//     bytes: a producer warp streams one tensor-map box per 256-weight
//     column and the x slices into a ring; consumer warp w decodes column w
//     of each 8-column unit, and the 8 warps' row sums meet in shared
//     memory once per tile.  IQ4_NL / IQ4_XS look each code up in a 16-entry
//     fp32 table (16 distinct banks: conflict-free); IQ3_S / IQ2_XXS join
//     grid and sign bytes with one byte permute per weight, from compact
//     grid tables in lane copies (or zero-interleaved rows when a codebook
//     byte is 128 or more).  The consumers build the tables while the
//     producer's first copies are in flight.
//   * qg_gemv_cb_kernel, the other rows: the 8 warps of a CTA on eighths of
//     K read the block fields directly with 16-bit loads (every field of
//     these layouts starts at an even byte), those of kDepth sub-blocks per
//     lane before any is decoded; x through the read-only cache.
#include <type_traits>

#include "launch_common.cuh"

namespace qg {
namespace cb {

constexpr int kIQ4NL = QG_CB_IQ4_NL, kIQ4XS = QG_CB_IQ4_XS, kIQ3S = QG_CB_IQ3_S, kIQ2XXS = QG_CB_IQ2_XXS;

__host__ __device__ constexpr int unit_bytes(int f) {  // bytes per 256 weights
    return f == kIQ4NL ? 144 : f == kIQ4XS ? 136 : f == kIQ3S ? 110 : 66;
}

__device__ __forceinline__ uint32_t ld16(const uint8_t* p) {
    return static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p)));
}
__device__ __forceinline__ uint32_t ld32e(const uint8_t* p) {  // 4 bytes at an even address
    return ld16(p) | (ld16(p + 2) << 16);
}

// Codebook in shared memory.
union Table {
    float iq4[16];
    uint32_t iq3s[512];
    uint2 iq2[256];
};

// The raw fields of one 32-weight sub-block, loaded before any of them is
// decoded so that a lane can keep several sub-blocks' loads in flight.
struct Raw {
    uint32_t r[6];
};

// Load the fields of sub-block sb of a row (row = the row's first byte).
// Field positions: see the oracle's decoders (page 3).
template <int F>
__device__ __forceinline__ void load_sub(const uint8_t* row, int64_t sb, Raw& R) {
    if constexpr (F == kIQ4NL) {
        // 18-byte block: d, then byte i = code of weight i (low) | weight i+16 (high)
        const uint8_t* blk = row + 18 * sb;
        R.r[0] = ld16(blk);
#pragma unroll
        for (int i = 0; i < 4; ++i) R.r[1 + i] = ld32e(blk + 2 + 4 * i);
    } else if constexpr (F == kIQ4XS) {
        // 136 bytes per 256: d, s high bits (u16 @2), s low nibbles @4, codes @8
        const int j = static_cast<int>(sb & 7);
        const uint8_t* u = row + 136 * (sb >> 3);
        R.r[0] = ld16(u) | (ld16(u + 2) << 16);
        R.r[1] = ld32e(u + 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) R.r[2 + i] = ld32e(u + 8 + 16 * j + 4 * i);
    } else if constexpr (F == kIQ3S) {
        // 110 bytes: d, index low bytes @2, 9th bits @66, sign bits @74, s nibbles @106
        const int j = static_cast<int>(sb & 7);
        const uint8_t* u = row + 110 * (sb >> 3);
        R.r[0] = ld16(u) | (ld16(u + 106 + 2 * (j >> 2)) << 16);
        R.r[1] = ld32e(u + 2 + 8 * j);
        R.r[2] = ld32e(u + 6 + 8 * j);
        R.r[3] = ld16(u + 66 + (j & ~1));
        R.r[4] = ld32e(u + 74 + 4 * j);
    } else {
        // 66 bytes: d, then per sub-block u32 grid indices + u32 (4 sign fields, s)
        const int j = static_cast<int>(sb & 7);
        const uint8_t* u = row + 66 * (sb >> 3);
        R.r[0] = ld16(u);
        R.r[1] = ld32e(u + 2 + 8 * j);
        R.r[2] = ld32e(u + 6 + 8 * j);
    }
}

// The 32 weights of sub-block sb from its loaded fields.
template <int F>
__device__ __forceinline__ void decode_sub(const Raw& R, int64_t sb, const Table& T, float (&w)[32]) {
    const int j = static_cast<int>(sb & 7);
    if constexpr (F == kIQ4NL || F == kIQ4XS) {
        float eff;
        if constexpr (F == kIQ4NL) {
            eff = h2f(R.r[0]);
        } else {
            const uint32_t sh = R.r[0] >> 16, sl = R.r[1];
            const int s = static_cast<int>(((sl >> (4 * j)) & 15u) | (((sh >> (2 * j)) & 3u) << 4));
            eff = h2f(R.r[0]) * static_cast<float>(s - 32);
        }
        constexpr int C = F == kIQ4NL ? 1 : 2;  // first code word
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t c = R.r[C + i];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                w[4 * i + e] = eff * T.iq4[(c >> (8 * e)) & 15u];
                w[16 + 4 * i + e] = eff * T.iq4[(c >> (8 * e + 4)) & 15u];
            }
        }
    } else if constexpr (F == kIQ3S) {
        const float d = h2f(R.r[0]);
        const float eff = d * static_cast<float>(1 + 2 * static_cast<int>((R.r[0] >> (16 + 4 * (j & 3))) & 15u));
        const uint32_t qh = (R.r[3] >> (8 * (j & 1))) & 0xFFu, sg = R.r[4];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const uint32_t idx = (((g < 4 ? R.r[1] : R.r[2]) >> (8 * (g & 3))) & 0xFFu) | (((qh >> g) & 1u) << 8);
            const uint32_t r = T.iq3s[idx];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float m = eff * static_cast<float>((r >> (8 * e)) & 0xFFu);
                w[4 * g + e] = ((sg >> (4 * g + e)) & 1u) ? -m : m;
            }
        }
    } else {
        const uint32_t aux0 = R.r[1], aux1 = R.r[2];
        const float eff = h2f(R.r[0]) * (0.5f + static_cast<float>(aux1 >> 28)) * 0.25f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint2 r = T.iq2[(aux0 >> (8 * g)) & 0xFFu];
            const uint32_t seven = (aux1 >> (7 * g)) & 0x7Fu;
            const uint32_t s8 = seven | ((__popc(seven) & 1u) << 7);  // implied eighth sign: even count
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float m = eff * static_cast<float>(((e < 4 ? r.x : r.y) >> (8 * (e & 3))) & 0xFFu);
                w[8 * g + e] = ((s8 >> e) & 1u) ? -m : m;
            }
        }
    }
}

// IQ4_NL / IQ4_XS sub-block as the 32 table values v and the sub-block's
// eff (weight = eff * v), for sums taken as eff * sum(v * x).
template <int F>
__device__ __forceinline__ void decode_sub_iq4_factored(const Raw& R, int64_t sb, const Table& T, float (&w)[32],
                                                        float& eff) {
    const int j = static_cast<int>(sb & 7);
    if constexpr (F == kIQ4NL) {
        eff = h2f(R.r[0]);
    } else {
        const uint32_t sh = R.r[0] >> 16, sl = R.r[1];
        const int s = static_cast<int>(((sl >> (4 * j)) & 15u) | (((sh >> (2 * j)) & 3u) << 4));
        eff = h2f(R.r[0]) * static_cast<float>(s - 32);
    }
    constexpr int C = F == kIQ4NL ? 1 : 2;  // first code word
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c = R.r[C + i];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            w[4 * i + e] = T.iq4[(c >> (8 * e)) & 15u];
            w[16 + 4 * i + e] = T.iq4[(c >> (8 * e + 4)) & 15u];
        }
    }
}

// Codebook -> shared memory, by threads tid = 0..nt-1 (the whole CTA by
// default).
template <int F>
__device__ void load_table(const void* book, Table& T, int tid = threadIdx.x, int nt = blockDim.x) {
    if constexpr (F == kIQ4NL || F == kIQ4XS) {
        const int8_t* t = static_cast<const int8_t*>(book);
        for (int i = tid; i < 16; i += nt) T.iq4[i] = static_cast<float>(t[i]);
    } else if constexpr (F == kIQ3S) {
        const uint32_t* t = static_cast<const uint32_t*>(book);
        for (int i = tid; i < 512; i += nt) T.iq3s[i] = t[i];
    } else {
        const uint2* t = static_cast<const uint2*>(book);
        for (int i = tid; i < 256; i += nt) T.iq2[i] = t[i];
    }
}

constexpr int kDepth = 4;  // consecutive sub-blocks a lane loads before decoding

// CTA = 32 rows (lane = row) x 8 warps; warp w takes the row's sub-blocks
// [w*K/256, (w+1)*K/256) (K/32 sub-blocks split evenly), so x loads are
// warp-wide broadcasts and each lane reads a contiguous stretch of its row.
// The 8 warps' partial sums meet in shared memory.
template <int F, int MT>
__global__ void __launch_bounds__(256) qg_gemv_cb_kernel(const uint8_t* __restrict__ W, const void* __restrict__ book,
                                                      const float* __restrict__ X, float* __restrict__ Y, int M,
                                                      int64_t N, int64_t K) {
    __shared__ Table T;
    __shared__ float red[8][MT][32];
    load_table<F>(book, T);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t per = K / 256;  // sub-blocks per warp
    const int64_t pitch = (K / 256) * unit_bytes(F);
    const int64_t ntiles = (N + 31) / 32;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t n = tile * 32 + lane;
        const bool live = n < N;
        const uint8_t* row = W + (live ? n : N - 1) * pitch;  // rows past N read row N-1, unused
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        const int64_t sb_end = (warp + 1) * per;
        for (int64_t sb0 = warp * per; sb0 < sb_end; sb0 += kDepth) {
            Raw R[kDepth];
#pragma unroll
            for (int p = 0; p < kDepth; ++p)
                if (sb0 + p < sb_end) load_sub<F>(row, sb0 + p, R[p]);
#pragma unroll
            for (int p = 0; p < kDepth; ++p) {
                const int64_t sb = sb0 + p;
                if (sb >= sb_end) break;
                float w[32];
                decode_sub<F>(R[p], sb, T, w);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (MT == 1 || m < M) {
                        const float4* xp = reinterpret_cast<const float4*>(X + m * K + 32 * sb);
                        float s = 0.f;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 x = __ldg(xp + q);
                            s = fmaf(w[4 * q], x.x, s);
                            s = fmaf(w[4 * q + 1], x.y, s);
                            s = fmaf(w[4 * q + 2], x.z, s);
                            s = fmaf(w[4 * q + 3], x.w, s);
                        }
                        acc[m] += s;
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) red[warp][m][lane] = acc[m];
        __syncthreads();
        for (int t = threadIdx.x; t < MT * 32; t += blockDim.x) {
            const int m = t >> 5, r = t & 31;
            const int64_t nn = tile * 32 + r;
            if ((MT == 1 || m < M) && nn < N) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) v += red[w][m][r];
                Y[m * N + nn] = v;
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ TMA-ring kernel
// The same decode (used for IQ4_NL and IQ4_XS) fed like the Q4_K / IQ3 GEMV: a producer warp streams each
// unit (32 rows x 8 columns of 256 weights) into a shared-memory ring with
// one 2D tensor-map box per column (the column's bytes from their offset
// rounded down to 16; every unit starts 16-byte aligned, as 8 columns of any
// of these formats are a multiple of 16 bytes) and the unit's x slice with a
// bulk copy; consumer warp w decodes column w, one row per lane, reading its
// box row with 16-byte loads (box rows 144 or 80 bytes apart: 8 consecutive
// lanes hit 8 distinct bank groups) and realigning it in registers.
template <int F>
struct Box {
    static constexpr int kUB = unit_bytes(F);
    static constexpr int kBox = F == kIQ2XXS ? 80 : 144;  // >= kUB + the largest in-box offset
    static constexpr int kWords = kBox / 4;
};

// Fields of sub-block j of a unit held as words v (v[k] = unit bytes 4k..4k+3);
// the positions of load_sub, every field at an even byte.
template <int B>
__device__ __forceinline__ uint32_t f16at(const uint32_t* v) {
    return (v[B >> 2] >> (8 * (B & 3))) & 0xFFFFu;
}
template <int B>
__device__ __forceinline__ uint32_t f32at(const uint32_t* v) {
    return (B & 3) ? __funnelshift_r(v[B >> 2], v[(B >> 2) + 1], 8 * (B & 3)) : v[B >> 2];
}
template <int F, int J>
__device__ __forceinline__ void raw_from_words(const uint32_t* v, Raw& R) {
    if constexpr (F == kIQ4NL) {
        R.r[0] = f16at<18 * J>(v);
        R.r[1] = f32at<18 * J + 2>(v);
        R.r[2] = f32at<18 * J + 6>(v);
        R.r[3] = f32at<18 * J + 10>(v);
        R.r[4] = f32at<18 * J + 14>(v);
    } else if constexpr (F == kIQ4XS) {
        R.r[0] = f32at<0>(v);
        R.r[1] = f32at<4>(v);
        R.r[2] = f32at<8 + 16 * J>(v);
        R.r[3] = f32at<12 + 16 * J>(v);
        R.r[4] = f32at<16 + 16 * J>(v);
        R.r[5] = f32at<20 + 16 * J>(v);
    } else if constexpr (F == kIQ3S) {
        R.r[0] = f16at<0>(v) | (f16at<106 + 2 * (J >> 2)>(v) << 16);
        R.r[1] = f32at<2 + 8 * J>(v);
        R.r[2] = f32at<6 + 8 * J>(v);
        R.r[3] = f16at<66 + (J & ~1)>(v);
        R.r[4] = f32at<74 + 4 * J>(v);
    } else {
        R.r[0] = f16at<0>(v);
        R.r[1] = f32at<2 + 8 * J>(v);
        R.r[2] = f32at<6 + 8 * J>(v);
    }
}

// One lane's row of one column, unit bytes OFF bytes into the box row, as
// NV aligned words (v[k] = unit bytes 4k..4k+3).
template <int F>
constexpr int row_words() { return (Box<F>::kUB + 3) / 4 + 1; }
template <int F, int OFF>
__device__ __forceinline__ void load_row_words(const uint8_t* boxrow, uint32_t (&v)[row_words<F>()]) {
    constexpr int NW = Box<F>::kWords, W0 = OFF >> 2, SH = 8 * (OFF & 3);
    uint32_t a[NW + 1];
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
        const uint4 t = *reinterpret_cast<const uint4*>(boxrow + 16 * i);
        a[4 * i] = t.x; a[4 * i + 1] = t.y; a[4 * i + 2] = t.z; a[4 * i + 3] = t.w;
    }
    a[NW] = 0u;  // past the box: only ever the unused top bytes of the last word
#pragma unroll
    for (int k = 0; k < row_words<F>(); ++k) {
        const int i0 = W0 + k < NW ? W0 + k : NW, i1 = W0 + k + 1 < NW ? W0 + k + 1 : NW;
        v[k] = SH ? __funnelshift_r(a[i0], a[i1], SH) : a[i0];
    }
}

// IQ4_NL / IQ4_XS: one lane's row of one column against MT tokens of x (xs:
// the column's 256 x values of token 0; tokens 2048 floats apart).
template <int F, int MT>
__device__ __forceinline__ void cb_iq4_column(const uint32_t (&v)[row_words<F>()], const float* xs, const Table& T,
                                              int M, float (&acc)[MT]) {
    auto sub = [&](auto jc) {
        constexpr int J = decltype(jc)::value;
        Raw R;
        raw_from_words<F, J>(v, R);
        float w[32];
        float eff = 1.f;
        decode_sub_iq4_factored<F>(R, J, T, w, eff);  // eff applied to the sub-block's sum
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (MT == 1 || m < M) {
                const float4* xp = reinterpret_cast<const float4*>(xs + m * 2048 + 32 * J);
                float s = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 x = xp[q];
                    s = fmaf(w[4 * q], x.x, s);
                    s = fmaf(w[4 * q + 1], x.y, s);
                    s = fmaf(w[4 * q + 2], x.z, s);
                    s = fmaf(w[4 * q + 3], x.w, s);
                }
                acc[m] = fmaf(eff, s, acc[m]);
            }
        }
    };
    sub(std::integral_constant<int, 0>{});
    sub(std::integral_constant<int, 1>{});
    sub(std::integral_constant<int, 2>{});
    sub(std::integral_constant<int, 3>{});
    sub(std::integral_constant<int, 4>{});
    sub(std::integral_constant<int, 5>{});
    sub(std::integral_constant<int, 6>{});
    sub(std::integral_constant<int, 7>{});
}

// ------------------------------------------------ grid formats on the ring
// IQ3_S and IQ2_XXS decode as the IQ3 GEMV does: the codebook's rows are
// expanded with zero bytes, so that one byte permute per weight puts the
// grid byte at bits 0-7 and its sign byte (0x80 when negative) at bits
// 24-31 of an fp32: the exact subnormal +-g * 2^-149, against x pre-scaled
// by 2^88 (cb_stage_x); the sub-block's eff * 2^61 undoes the scaling.
//   IQ3_S    entry i (4 weights) -> [g0,0,g1,0][g2,0,g3,0]          512 x 8 bytes
//   IQ2_XXS  entry i (8 weights) -> [g0,0,g1,0] ... [g6,0,g7,0]     256 x 16 bytes,
//            then the sign bytes of each 7-bit field (the eighth sign
//            its parity: an even count of negatives)                128 x 8 bytes
constexpr int kGridTabBytes = 5120;
// Compact tables are kept in kGridCopies copies, entry i of copy c at
// i * kGridCopies + c, lane L reading copy L & 7: the 32 rows' random
// lookups then meet at most 4 to a copy instead of 32 to one table (a
// capture counted 4.7 wavefronts per lookup with one copy).
constexpr int kGridCopies = 8;

// Sign bytes of four sign bits: bit k of nib -> bit 8k+7 (one multiply
// places bit k at k, k+7, k+14, k+21 and k+28, which never collide).
__device__ __forceinline__ uint32_t sign_bytes(uint32_t nib) { return (nib * 0x10204081u) & 0x80808080u; }

// [b0, 0, b1, 0] of the low two bytes of w
__device__ __forceinline__ uint32_t spread2(uint32_t w) { return (w & 0xFFu) | ((w & 0xFF00u) << 8); }

// Nonzero in every participating thread when pred is nonzero in any of
// the nt threads (a multiple of 32) that meet on named barrier id.
__device__ __forceinline__ bool named_barrier_or(int id, int nt, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nt) : "memory");
    return r != 0u;
}

// Loads the codebook; returns true (the same in every calling thread) when
// every codebook byte is below 128.  Then the table keeps the codebook's
// own rows (IQ3_S 512 x 4 bytes, IQ2_XXS 256 x 8 bytes, half the bytes per
// gather) in kGridCopies lane copies, IQ2_XXS's sign table after them, and
// the permute takes the zero bytes from the sign-replicate of the grid byte
// itself (its top bit is 0); otherwise the rows are expanded as above, one
// copy.  Threads tid = 0..nt-1, all of which call it, meet on named barrier
// bar (nt a multiple of 32); the caller synchronises them again before the
// table is read.
template <int F>
__device__ bool load_grid_table(const void* book, uint8_t* gt, int tid, int nt, int bar) {
    const uint32_t* w = static_cast<const uint32_t*>(book);
    uint32_t high = 0;
    for (int i = tid; i < 512; i += nt) high |= w[i];  // both formats: 2 KB
    const bool compact = !named_barrier_or(bar, nt, (high & 0x80808080u) != 0u);
    if (compact) {
        if constexpr (F == kIQ3S) {
            uint32_t* t = reinterpret_cast<uint32_t*>(gt);
            for (int i = tid; i < 512 * kGridCopies; i += nt) t[i] = w[i / kGridCopies];
        } else {
            uint2* t = reinterpret_cast<uint2*>(gt);
            const uint2* w2 = static_cast<const uint2*>(book);
            for (int i = tid; i < 256 * kGridCopies; i += nt) t[i] = w2[i / kGridCopies];
            uint2* sg = reinterpret_cast<uint2*>(gt + 256 * 8 * kGridCopies);
            for (int i = tid; i < 128 * kGridCopies; i += nt) {
                const uint32_t s7 = static_cast<uint32_t>(i / kGridCopies);
                const uint32_t s8 = s7 | ((__popc(s7) & 1u) << 7);
                sg[i] = make_uint2(sign_bytes(s8 & 15u), sign_bytes(s8 >> 4));
            }
        }
        return true;
    }
    if constexpr (F == kIQ3S) {
        const uint32_t* t = static_cast<const uint32_t*>(book);
        uint2* e = reinterpret_cast<uint2*>(gt);
        for (int i = tid; i < 512; i += nt) e[i] = make_uint2(spread2(t[i]), spread2(t[i] >> 16));
    } else {
        const uint2* t = static_cast<const uint2*>(book);
        uint4* e = reinterpret_cast<uint4*>(gt);
        for (int i = tid; i < 256; i += nt) {
            const uint2 g = t[i];
            e[i] = make_uint4(spread2(g.x), spread2(g.x >> 16), spread2(g.y), spread2(g.y >> 16));
        }
        uint2* sg = reinterpret_cast<uint2*>(gt + 4096);
        for (int i = tid; i < 128; i += nt) {
            const uint32_t s8 = static_cast<uint32_t>(i) | ((__popc(i) & 1u) << 7);
            sg[i] = make_uint2(sign_bytes(s8 & 15u), sign_bytes(s8 >> 4));
        }
    }
    return false;
}

// Signed grid value: byte P (0 or 2) of the expanded word g, sign byte K of s.
template <int P, int K>
__device__ __forceinline__ float grid_val(uint32_t g, uint32_t s) {
    return __uint_as_float(prmt(g, s, static_cast<uint32_t>(P) | (1u << 4) | (1u << 8) | ((4u + K) << 12)));
}
// The same from a compact row word (bytes below 128): byte P at bits 0-7,
// bits 8-23 the replicated top bit of byte P (0), sign byte K at 24-31.
template <int P, int K>
__device__ __forceinline__ float grid_val_c(uint32_t g, uint32_t s) {
    constexpr uint32_t rep = 8u | P;
    return __uint_as_float(prmt(g, s, static_cast<uint32_t>(P) | (rep << 4) | (rep << 8) | ((4u + K) << 12)));
}

// IQ3_S / IQ2_XXS: one lane's row of one column against MT tokens of x
// (pre-scaled by 2^88; tokens 2048 floats apart).  With RESCALE the
// column's sums are formed apart and multiplied by e2[m] before they join
// acc (a token whose column cb_stage_x rescaled).
template <int F, int MT, bool RESCALE, bool COMPACT>
__device__ __forceinline__ void cb_grid_column(const uint32_t (&v)[row_words<F>()], const float* xs,
                                               const uint8_t* gt, int M, const float (&e2)[MT], float (&acc)[MT],
                                               uint32_t lc) {
    if constexpr (RESCALE && MT > 1) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                float a1[1] = {acc[m]};
                const float e1[1] = {e2[m]};
                cb_grid_column<F, 1, true, COMPACT>(v, xs + m * 2048, gt, 1, e1, a1, lc);
                acc[m] = a1[0];
            }
        }
        return;
    }
    float part[MT];
    float (&tgt)[MT] = RESCALE ? part : acc;
    if constexpr (RESCALE) {
#pragma unroll
        for (int m = 0; m < MT; ++m) part[m] = 0.f;
    }
    // four weights: expanded words ga = [g0,0,g1,0], gb = [g2,0,g3,0], or
    // (COMPACT) one word ga = [g0 g1 g2 g3]
    auto four = [&](uint32_t ga, uint32_t gb, uint32_t sgn, const float* xq, f2 (&dot)[MT]) {
        f2 w01, w23;
        if constexpr (COMPACT) {
            w01 = f2{grid_val_c<0, 0>(ga, sgn), grid_val_c<1, 1>(ga, sgn)};
            w23 = f2{grid_val_c<2, 2>(ga, sgn), grid_val_c<3, 3>(ga, sgn)};
        } else {
            w01 = f2{grid_val<0, 0>(ga, sgn), grid_val<2, 1>(ga, sgn)};
            w23 = f2{grid_val<0, 2>(gb, sgn), grid_val<2, 3>(gb, sgn)};
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (MT == 1 || m < M) {
                const float4 x = *reinterpret_cast<const float4*>(xq + m * 2048);
                ffma2(dot[m], w01, f2{x.x, x.y});
                ffma2(dot[m], w23, f2{x.z, x.w});
            }
        }
    };
    auto sub = [&](auto jc) {
        constexpr int J = decltype(jc)::value;
        Raw R;
        raw_from_words<F, J>(v, R);
        f2 dot[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) dot[m] = f2{0.f, 0.f};
        float eff61;
        if constexpr (F == kIQ3S) {
            // eff = d*(1+2s); 9-bit indices (low byte + one high bit); one sign bit per weight
            const uint32_t sc = (R.r[0] >> (16 + 4 * (J & 3))) & 15u;
            eff61 = h2f(R.r[0]) * static_cast<float>(1u + 2u * sc) * 0x1p61f;
            const uint32_t qh = (R.r[3] >> (8 * (J & 1))) & 0xFFu, sg = R.r[4];
            // the ninth index bits, bit k of each half of qh moved to bit 0
            // of byte k (no two shifted copies overlap), so that one byte
            // permute per group joins an index's two bytes: [low, high, 0, 0]
            const uint32_t hb[2] = {((qh & 15u) * 0x00204081u) & 0x01010101u, ((qh >> 4) * 0x00204081u) & 0x01010101u};
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                constexpr uint32_t kZero = 0xCu;  // replicate bit 7 of byte 0 of hb (clear): a zero byte
                const uint32_t idx = prmt(g < 4 ? R.r[1] : R.r[2], hb[g >> 2],
                                          static_cast<uint32_t>(g & 3) | ((4u + (g & 3)) << 4) | (kZero << 8) |
                                              (kZero << 12));
                const uint32_t sgn = sign_bytes((sg >> (4 * g)) & 15u);
                if constexpr (COMPACT) {
                    four(reinterpret_cast<const uint32_t*>(gt)[idx * kGridCopies + lc], 0u, sgn, xs + 32 * J + 4 * g, dot);
                } else {
                    const uint2 ge = reinterpret_cast<const uint2*>(gt)[idx];
                    four(ge.x, ge.y, sgn, xs + 32 * J + 4 * g, dot);
                }
            }
        } else {
            // eff = d*(0.5+s)*0.25; four 8-weight groups, each a grid index byte and a 7-bit sign field
            const uint32_t aux0 = R.r[1], aux1 = R.r[2];
            eff61 = h2f(R.r[0]) * (0.5f + static_cast<float>(aux1 >> 28)) * (0.25f * 0x1p61f);
            const uint2* sgt = reinterpret_cast<const uint2*>(gt + (COMPACT ? 256 * 8 * kGridCopies : 4096));
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint32_t idx = (aux0 >> (8 * g)) & 0xFFu;
                const uint32_t s7 = (aux1 >> (7 * g)) & 0x7Fu;
                const uint2 sgn = COMPACT ? sgt[s7 * kGridCopies + lc] : sgt[s7];
                if constexpr (COMPACT) {
                    const uint2 ge = reinterpret_cast<const uint2*>(gt)[idx * kGridCopies + lc];
                    four(ge.x, 0u, sgn.x, xs + 32 * J + 8 * g, dot);
                    four(ge.y, 0u, sgn.y, xs + 32 * J + 8 * g + 4, dot);
                } else {
                    const uint4 ge = reinterpret_cast<const uint4*>(gt)[idx];
                    four(ge.x, ge.y, sgn.x, xs + 32 * J + 8 * g, dot);
                    four(ge.z, ge.w, sgn.y, xs + 32 * J + 8 * g + 4, dot);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (MT == 1 || m < M) tgt[m] = fmaf(eff61, dot[m].x + dot[m].y, tgt[m]);
    };
    sub(std::integral_constant<int, 0>{});
    sub(std::integral_constant<int, 1>{});
    sub(std::integral_constant<int, 2>{});
    sub(std::integral_constant<int, 3>{});
    sub(std::integral_constant<int, 4>{});
    sub(std::integral_constant<int, 5>{});
    sub(std::integral_constant<int, 6>{});
    sub(std::integral_constant<int, 7>{});
    if constexpr (RESCALE) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (MT == 1 || m < M) acc[m] = fmaf(part[m], e2[m], acc[m]);
    }
}

// Per-warp x preparation of one column (256 values per token, tokens 2048
// floats apart) for the grid formats: scaled in place by 2^88; a token
// whose largest |x| lies outside [2^-24, 2^39) is also scaled by 2^-e (e
// the exponent of its largest |x|, clamped to [-100, 100]), e2[m] = 2^e
// then (1 otherwise), and the return value, the same in every lane, says
// whether any token was.  Callers fence the written x before the slot's
// next copy.
template <int MT>
__device__ __forceinline__ bool cb_stage_x(float* xs, int M, int lane, float (&e2)[MT]) {
    bool rescaled = false;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        e2[m] = 1.f;
        if (MT == 1 || m < M) {
            float* xp = xs + m * 2048 + lane * 8;
            float4 a = *reinterpret_cast<const float4*>(xp);
            float4 b = *reinterpret_cast<const float4*>(xp + 4);
            const float mx = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                                   fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
            const uint32_t top = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
            const uint32_t be = top >> 23;
            if (top != 0u && (be < kXExpLo || be >= kXExpHi)) {  // the same in every lane
                const int e = min(max(static_cast<int>(be) - 127, -100), 100);
                const float sc = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
                a = make_float4(a.x * sc, a.y * sc, a.z * sc, a.w * sc);
                b = make_float4(b.x * sc, b.y * sc, b.z * sc, b.w * sc);
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

constexpr int kCbCols = 8;        // columns per unit = consumer warps
constexpr int kCbMaxStages = 4;
// Dynamic shared memory: barriers at 0, the codebook at 128 (IQ4: the 16
// table values; grid formats: their tables), the warps' row sums after it,
// the ring from 10240.
constexpr int kCbTable0 = 128;
static_assert(sizeof(Table) <= kGridTabBytes, "codebook slot");
// The codebook region: IQ4's Table or an expanded grid table (at most
// kGridTabBytes), or a compact grid table in kGridCopies copies (IQ2_XXS
// with its sign table); then the row sums (up to 4 tokens), then the ring.
__host__ __device__ constexpr int cb_table_bytes(int F) {
    return F == kIQ3S ? 512 * 4 * kGridCopies : F == kIQ2XXS ? (256 + 128) * 8 * kGridCopies : kGridTabBytes;
}
__host__ __device__ constexpr int cb_red0(int F) { return kCbTable0 + cb_table_bytes(F); }
__host__ __device__ constexpr int cb_ring0(int F) { return (cb_red0(F) + kCbCols * 4 * 32 * 4 + 1023) / 1024 * 1024; }
static_assert(cb_table_bytes(kIQ3S) >= kGridTabBytes && cb_table_bytes(kIQ2XXS) >= kGridTabBytes, "expanded tables fit");
__host__ __device__ constexpr int cb_stage_bytes(int F, int MT) {
    return kCbCols * 32 * (F == kIQ2XXS ? 80 : 144) + MT * kCbCols * 1024;
}

template <int F, int MT, int MINB>
__global__ void __launch_bounds__(kCbCols * 32 + 32, MINB)
    qg_gemv_cb_tma_kernel(const __grid_constant__ CUtensorMap tmW, const void* __restrict__ book,
                       const float* __restrict__ X, float* __restrict__ Y, int M, int64_t N, int64_t K, int stages,
                       unsigned* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Table& T = *reinterpret_cast<Table*>(smem + kCbTable0);
    float (*red)[MT][32] = reinterpret_cast<float (*)[MT][32]>(smem + cb_red0(F));
    static_assert(MT <= 4 && cb_red0(F) + kCbCols * MT * 32 * 4 <= cb_ring0(F), "row-sum slot");
    constexpr int kBox = Box<F>::kBox, kUB = Box<F>::kUB;
    constexpr int kColBytes = 32 * kBox;
    constexpr int kSB = cb_stage_bytes(F, MT);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kCbMaxStages;
    uint8_t* ring = smem + cb_ring0(F);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = static_cast<int>(K / 256);
    const int nchunks = (nb + kCbCols - 1) / kCbCols;
    const int64_t ntiles = (N + 31) / 32;
    const int64_t my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t U = my_tiles * nchunks;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCbCols);
        }
        fence_mbar_init();
    }
    constexpr bool kGrid = F == kIQ3S || F == kIQ2XXS;
    __syncthreads();  // the barriers are initialised

    // The producer starts the weight stream at once; the consumer warps
    // build the codebook table meanwhile (named barriers 2 and 3 among
    // them), so its global loads overlap the first copies.
    if (warp == kCbCols) {
        // ---------------- producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            int s = 0, c = 0;
            uint32_t round = 0;
            int64_t tile = blockIdx.x;
            for (int64_t u = 0; u < U; ++u) {
                if (u >= stages) mbar_wait_bounded(&empty[s], (round - 1) & 1u, status);
                const int kc = min(kCbCols, nb - c * kCbCols);
                uint8_t* st = ring + s * kSB;
                mbar_arrive_expect_tx(&full[s], kc * kColBytes + M * kc * 1024);
                for (int b = 0; b < kc; ++b)
                    tma_load_2d(st + b * kColBytes, &tmW, ((c * kCbCols + b) * kUB) & ~15,
                                static_cast<int>(tile * 32), &full[s], pol_w);
                for (int m = 0; m < M; ++m)
                    bulk_g2s(st + kCbCols * kColBytes + m * kCbCols * 1024,
                             X + m * K + static_cast<int64_t>(c) * kCbCols * 256, kc * 1024, &full[s], pol_x);
                if (++s == stages) {
                    s = 0;
                    ++round;
                }
                if (++c == nchunks) {
                    c = 0;
                    tile += gridDim.x;
                }
            }
        }
        return;
    }

    // ---------------- consumers: warp = column, lane = row
    bool compact = false;  // grid formats: codebook bytes all below 128 (the same in every consumer)
    if constexpr (kGrid)
        compact = load_grid_table<F>(book, smem + kCbTable0, threadIdx.x, kCbCols * 32, 3);
    else
        load_table<F>(book, T, threadIdx.x, kCbCols * 32);
    named_barrier_sync<kCbCols * 32>(2);
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    int s = 0, c = 0;
    uint32_t phase = 0;
    int64_t tile = blockIdx.x;
    for (int64_t u = 0; u < U; ++u) {
        const int kc = min(kCbCols, nb - c * kCbCols);
        const uint8_t* st = ring + s * kSB;
        mbar_wait_bounded(&full[s], phase, status);
        if (warp < kc) {
            const uint8_t* boxrow = st + warp * kColBytes + lane * kBox;
            float* xs = reinterpret_cast<float*>(const_cast<uint8_t*>(st) + kCbCols * kColBytes) + warp * 256;
            // the column's offset in its box: (kUB * column) mod 16, and
            // 8 * kUB is a multiple of 16
            uint32_t v[row_words<F>()];
            switch ((warp * kUB) & 15) {
#define QG_CB_COL(O) \
    case O: load_row_words<F, O>(boxrow, v); break;
                QG_CB_COL(0) QG_CB_COL(2) QG_CB_COL(4) QG_CB_COL(6)
                QG_CB_COL(8) QG_CB_COL(10) QG_CB_COL(12) QG_CB_COL(14)
#undef QG_CB_COL
                default: break;
            }
            if constexpr (kGrid) {
                float e2[MT];
                const bool rescaled = cb_stage_x<MT>(xs, M, lane, e2);
                __syncwarp();
                const uint8_t* gt = smem + kCbTable0;
                if (rescaled) {  // rare; the same in every lane
                    if (compact)
                        cb_grid_column<F, MT, true, true>(v, xs, gt, M, e2, acc, lane & 7);
                    else
                        cb_grid_column<F, MT, true, false>(v, xs, gt, M, e2, acc, lane & 7);
                } else if (compact) {
                    cb_grid_column<F, MT, false, true>(v, xs, gt, M, e2, acc, lane & 7);
                } else {
                    cb_grid_column<F, MT, false, false>(v, xs, gt, M, e2, acc, lane & 7);
                }
                fence_proxy_async_smem();  // x was written: order it before the slot's next copy
            } else {
                cb_iq4_column<F, MT>(v, xs, T, M, acc);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (c == nchunks - 1) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                red[warp][m][lane] = acc[m];
                acc[m] = 0.f;
            }
            named_barrier_sync<kCbCols * 32>(1);
            for (int t = threadIdx.x; t < MT * 32; t += kCbCols * 32) {
                const int m = t >> 5, r = t & 31;
                const int64_t nn = tile * 32 + r;
                if ((MT == 1 || m < M) && nn < N) {
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < kCbCols; ++w) v += red[w][m][r];
                    Y[m * N + nn] = v;
                }
            }
            named_barrier_sync<kCbCols * 32>(1);
        }
        if (++s == stages) {
            s = 0;
            phase ^= 1u;
        }
        if (++c == nchunks) {
            c = 0;
            tile += gridDim.x;
        }
    }
}

// The TMA path: every format whose rows are a multiple of 16 bytes (IQ4_NL
// always; IQ4_XS for even K/256; IQ3_S and IQ2_XXS for K/256 a multiple of
// 8).  Other rows take the direct-load kernel.
inline bool tma_ok(int F, int64_t K) { return ((K / 256) * unit_bytes(F)) % 16 == 0; }

template <int F, int MT, int MINB>
int launch_tma(const uint8_t* W, const void* book, const float* X, float* Y, int M, int64_t N, int64_t K,
               cudaStream_t s, unsigned* status, int dev, int sms) {
    static std::atomic<bool> attr_done[64];
    const int budget = std::min(kSmemPerCTA, kSmemPerSM / MINB - kSmemReserve) - cb_ring0(F);
    const int stages = std::min(kCbMaxStages, budget / cb_stage_bytes(F, MT));
    if (stages < 2) return QG_EINVAL;
    auto kern = qg_gemv_cb_tma_kernel<F, MT, MINB>;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 std::min(kSmemPerCTA, cb_ring0(F) + kCbMaxStages * cb_stage_bytes(F, MT))) !=
            cudaSuccess)
            return qg::cuda_fail(cudaGetLastError());
        attr_done[dev].store(true, std::memory_order_release);
    }
    CUtensorMap tm;
    const uint64_t pitch = static_cast<uint64_t>(K / 256) * unit_bytes(F);
    if (!encode_byte_rows(&tm, W, pitch, static_cast<uint64_t>(N), Box<F>::kBox, 32)) return qg::cuda_fail(cudaGetLastError());
    const int64_t ntiles = (N + 31) / 32;
    const int grid = static_cast<int>(std::min<int64_t>(ntiles, static_cast<int64_t>(sms) * MINB));
    const int64_t units_per_cta = (ntiles + grid - 1) / grid * ((K / 256 + kCbCols - 1) / kCbCols);
    const int st = static_cast<int>(std::min<int64_t>(stages, std::max<int64_t>(2, units_per_cta)));
    kern<<<grid, kCbCols * 32 + 32, cb_ring0(F) + st * cb_stage_bytes(F, MT), s>>>(tm, book, X, Y, M, N, K, st, status);
    return launch_status();
}

// Test-only: every sub-block's 32 values (exact), one thread per sub-block.
template <int F>
__global__ void __launch_bounds__(256) qg_dequant_cb_kernel(const uint8_t* __restrict__ W, const void* __restrict__ book,
                                                         float* __restrict__ out, int64_t N, int64_t K) {
    __shared__ Table T;
    load_table<F>(book, T);
    __syncthreads();
    const int64_t nsub = K / 32, pitch = (K / 256) * unit_bytes(F);
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= N * nsub) return;
    const int64_t n = i / nsub, sb = i % nsub;
    Raw R;
    load_sub<F>(W + n * pitch, sb, R);
    float w[32];
    decode_sub<F>(R, sb, T, w);
#pragma unroll
    for (int t = 0; t < 32; ++t) out[n * K + 32 * sb + t] = w[t];
}

template <int F>
int launch_t(const uint8_t* W, const void* book, const float* X, float* Y, int M, int64_t N, int64_t K,
             cudaStream_t s, unsigned* status) {
    const int dev = current_device();
    if (dev < 0) return qg::cuda_fail(cudaGetLastError());
    const int sms = sm_count(dev);
    if (sms <= 0) return qg::cuda_fail(cudaGetLastError());
    {
        if (tma_ok(F, K)) {
            // groups of at most 4 tokens, each streaming W once
            for (int m0 = 0; m0 < M; m0 += 4) {
                const int mg = std::min(4, M - m0);
                const float* Xg = X + static_cast<int64_t>(m0) * K;
                float* Yg = Y + static_cast<int64_t>(m0) * N;
                const int rc = mg == 1 ? launch_tma<F, 1, 2>(W, book, Xg, Yg, mg, N, K, s, status, dev, sms)
                                       : launch_tma<F, 4, 1>(W, book, Xg, Yg, mg, N, K, s, status, dev, sms);
                if (rc != QG_OK) return rc;
            }
            return QG_OK;
        }
    }
    const int blocks = static_cast<int>(std::min<int64_t>((N + 31) / 32, static_cast<int64_t>(sms) * 8));
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mg = std::min(8, M - m0);
        const float* Xg = X + static_cast<int64_t>(m0) * K;
        float* Yg = Y + static_cast<int64_t>(m0) * N;
        if (mg == 1)
            qg_gemv_cb_kernel<F, 1><<<blocks, 256, 0, s>>>(W, book, Xg, Yg, mg, N, K);
        else if (mg <= 4)
            qg_gemv_cb_kernel<F, 4><<<blocks, 256, 0, s>>>(W, book, Xg, Yg, mg, N, K);
        else
            qg_gemv_cb_kernel<F, 8><<<blocks, 256, 0, s>>>(W, book, Xg, Yg, mg, N, K);
        if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) return qg::cuda_fail(e);
    }
    return QG_OK;
}

template <int F>
int dequant_t(const uint8_t* W, const void* book, float* out, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t threads = N * (K / 32);
    qg_dequant_cb_kernel<F><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(W, book, out, N, K);
    return launch_status();
}

}  // namespace cb

int cb_unit_bytes(int format) { return cb::unit_bytes(format); }

int launch_gemv_cb(int format, const uint8_t* W, const void* book, const float* X, float* Y, int M, int64_t N,
                   int64_t K, cudaStream_t s, unsigned* status) {
    switch (format) {
        case QG_CB_IQ4_NL: return cb::launch_t<cb::kIQ4NL>(W, book, X, Y, M, N, K, s, status);
        case QG_CB_IQ4_XS: return cb::launch_t<cb::kIQ4XS>(W, book, X, Y, M, N, K, s, status);
        case QG_CB_IQ3_S: return cb::launch_t<cb::kIQ3S>(W, book, X, Y, M, N, K, s, status);
        case QG_CB_IQ2_XXS: return cb::launch_t<cb::kIQ2XXS>(W, book, X, Y, M, N, K, s, status);
        default: return QG_EINVAL;
    }
}

int launch_dequant_cb(int format, const uint8_t* W, const void* book, float* out, int64_t N, int64_t K,
                      cudaStream_t s) {
    switch (format) {
        case QG_CB_IQ4_NL: return cb::dequant_t<cb::kIQ4NL>(W, book, out, N, K, s);
        case QG_CB_IQ4_XS: return cb::dequant_t<cb::kIQ4XS>(W, book, out, N, K, s);
        case QG_CB_IQ3_S: return cb::dequant_t<cb::kIQ3S>(W, book, out, N, K, s);
        case QG_CB_IQ2_XXS: return cb::dequant_t<cb::kIQ2XXS>(W, book, out, N, K, s);
        default: return QG_EINVAL;
    }
}

}  // namespace qg
