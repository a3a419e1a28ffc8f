// GEMV (fp32 FMA) over page 3's other codebook formats: IQ4_NL, IQ4_XS,
// IQ3_S, IQ2_XXS (llama.cpp's codebook formats as trainable students: the
// format table, get_s, eff_np and encode).  weight = eff * v, v = codebook
// entry * sign; every value is exact in fp32.
//
// One lane per row (32 rows per CTA), the 8 warps of a CTA on eighths of K;
// the codebook sits in shared
// memory (IQ4: 16 fp32 values, which occupy 16 distinct banks, so any
// gather is conflict-free; IQ3_S: 512 x 4 bytes; IQ2_XXS: 256 x 8 bytes);
// x is read through the read-only cache (shared by all rows).  Block fields
// are read with 16-bit loads (every field of these layouts starts at an even
// byte), those of kDepth sub-blocks per lane before any is decoded, to keep
// enough bytes in flight.  Per row, the lanes' partial sums meet in a warp
// shuffle.
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

template <int F>
__device__ void load_table(const void* book, Table& T) {
    if constexpr (F == kIQ4NL || F == kIQ4XS) {
        const int8_t* t = static_cast<const int8_t*>(book);
        for (int i = threadIdx.x; i < 16; i += blockDim.x) T.iq4[i] = static_cast<float>(t[i]);
    } else if constexpr (F == kIQ3S) {
        const uint32_t* t = static_cast<const uint32_t*>(book);
        for (int i = threadIdx.x; i < 512; i += blockDim.x) T.iq3s[i] = t[i];
    } else {
        const uint2* t = static_cast<const uint2*>(book);
        for (int i = threadIdx.x; i < 256; i += blockDim.x) T.iq2[i] = t[i];
    }
}

constexpr int kDepth = 4;  // consecutive sub-blocks a lane loads before decoding

// CTA = 32 rows (lane = row) x 8 warps; warp w takes the row's sub-blocks
// [w*K/256, (w+1)*K/256) (K/32 sub-blocks split evenly), so x loads are
// warp-wide broadcasts and each lane reads a contiguous stretch of its row.
// The 8 warps' partial sums meet in shared memory.
template <int F, int MT>
__global__ void __launch_bounds__(256) gemv_cb_kernel(const uint8_t* __restrict__ W, const void* __restrict__ book,
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

// Test-only: every sub-block's 32 values (exact), one thread per sub-block.
template <int F>
__global__ void __launch_bounds__(256) dequant_cb_kernel(const uint8_t* __restrict__ W, const void* __restrict__ book,
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
             cudaStream_t s) {
    const int dev = current_device();
    if (dev < 0) return QG_ECUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return QG_ECUDA;
    const int blocks = static_cast<int>(std::min<int64_t>((N + 31) / 32, static_cast<int64_t>(sms) * 8));
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mg = std::min(8, M - m0);
        const float* Xg = X + static_cast<int64_t>(m0) * K;
        float* Yg = Y + static_cast<int64_t>(m0) * N;
        if (mg == 1)
            gemv_cb_kernel<F, 1><<<blocks, 256, 0, s>>>(W, book, Xg, Yg, mg, N, K);
        else if (mg <= 4)
            gemv_cb_kernel<F, 4><<<blocks, 256, 0, s>>>(W, book, Xg, Yg, mg, N, K);
        else
            gemv_cb_kernel<F, 8><<<blocks, 256, 0, s>>>(W, book, Xg, Yg, mg, N, K);
        if (cudaGetLastError() != cudaSuccess) return QG_ECUDA;
    }
    return QG_OK;
}

template <int F>
int dequant_t(const uint8_t* W, const void* book, float* out, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t threads = N * (K / 32);
    dequant_cb_kernel<F><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(W, book, out, N, K);
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

}  // namespace cb

int cb_unit_bytes(int format) { return cb::unit_bytes(format); }

int launch_gemv_cb(int format, const uint8_t* W, const void* book, const float* X, float* Y, int M, int64_t N,
                   int64_t K, cudaStream_t s) {
    switch (format) {
        case QG_CB_IQ4_NL: return cb::launch_t<cb::kIQ4NL>(W, book, X, Y, M, N, K, s);
        case QG_CB_IQ4_XS: return cb::launch_t<cb::kIQ4XS>(W, book, X, Y, M, N, K, s);
        case QG_CB_IQ3_S: return cb::launch_t<cb::kIQ3S>(W, book, X, Y, M, N, K, s);
        case QG_CB_IQ2_XXS: return cb::launch_t<cb::kIQ2XXS>(W, book, X, Y, M, N, K, s);
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
