// Batched Q4_K GEMM on the tcgen05 tensor cores (16 <= M <= 32 tokens).
//
//   Y[m][n] = sum_k w[n][k] * X[m][k]
//
// Only here the path is a dense contraction: a 128-row tile of W is
// dequantised (page 1 "Rewriting picoLM in Python", dequantize_q4_K:
// (d*sc)*q - dmin*mn, one fp32 rounding) and rounded to bf16 (RN) in shared
// memory; X is rounded to bf16 likewise; tcgen05.mma (kind::f16, bf16 x bf16,
// fp32 accumulation in tensor memory) computes D[row][token] = W_tile X^T
// (W rows on the MMA's M=128 side, tokens on its N=16/32 side).
//
// CTA roles (192 threads):
//   warps 0-3  dequantise W (thread t = tile row t) and X into the operand
//              stage, then drain the accumulator (tcgen05.ld) into Y;
//   warp 4     producer: cp.async.bulk of each row's 144-byte block and of
//              the fp32 x slice into a double-buffered raw stage;
//   warp 5     allocates tensor memory; lane 0 issues the MMAs and commits
//              them to mbarriers.
// Work: units (tile, k-block) in row-major order, split evenly over the grid
// (stream-K); a CTA's run over one tile is a "segment" whose partial sums are
// added into Y (zeroed first) with fp32 atomics.
//
// Operand layout (no swizzle, K-major): 8-row x 16-byte core matrices;
// core (row group i, k chunk j) at ((i * 32) + j) * 128 bytes, row r of the
// core at +16 r.  Adjacent k chunks are 128 bytes apart, adjacent row groups
// 4096 bytes apart.
#include <cuda_bf16.h>

#include <algorithm>

#include "gemv_kernel.cuh"
#include "launch.h"

namespace qg {
namespace tc {

constexpr int kTileRows = 128;
constexpr int kBlockBytes = 144;
constexpr int kThreads = 192;
constexpr int kRawW = kTileRows * kBlockBytes;     // 18432
constexpr int kRawX = 32 * 1024;                    // up to 32 tokens x 256 fp32
constexpr int kRawStage = kRawW + kRawX;            // 51200
constexpr int kOpA = kTileRows * 256 * 2;           // 65536: 128 rows x 256 k bf16
constexpr int kOpB = 32 * 256 * 2;                  // 16384: 32 tokens x 256 k bf16
constexpr int kRaw0 = 1024;
constexpr int kOpA0 = kRaw0 + 2 * kRawStage;        // 103424
constexpr int kOpB0 = kOpA0 + kOpA;                 // 168960
constexpr int kSmemTotal = kOpB0 + kOpB;            // 185344
constexpr int kTmemCols = 32;

// smem descriptor for tcgen05.mma: start address, leading (k) and stride
// (row group) byte offsets, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // version
    return d;  // base offset 0, layout type 0 (no swizzle)
}

// instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t instr_desc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<const uint32_t*>(&v);
}

// 32 fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Offset of the 16-byte chunk (row, k chunk j) in an operand buffer.
__device__ __forceinline__ uint32_t op_off(int row, int j) {
    return static_cast<uint32_t>((((row >> 3) * 32) + j) * 128 + (row & 7) * 16);
}

// Thread t: W tile row t, one 256-weight block -> 32 chunks of 8 bf16.
// Weights are formed exactly in fp32 ((d*sc)*q - dmin*mn with both products
// exact, one rounding) and then rounded to bf16.
__device__ __forceinline__ void dequant_row(const uint8_t* blk, uint8_t* opA, int t) {
    const uint4 h = *reinterpret_cast<const uint4*>(blk);
    const float d = h2f(h.x), dmin = h2f(h.x >> 16);
    uint32_t sc03, mn03, sc47, mn47;
    q4k_scale_min_words(h.y, h.z, h.w, sc03, mn03, sc47, mn47);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t scw = g < 2 ? sc03 : sc47, mnw = g < 2 ? mn03 : mn47;
        const float dl = d * byte_f(scw, (2 * g) & 3), ml = dmin * byte_f(mnw, (2 * g) & 3);
        const float dh = d * byte_f(scw, (2 * g + 1) & 3), mh = dmin * byte_f(mnw, (2 * g + 1) & 3);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint4 q = *reinterpret_cast<const uint4*>(blk + 16 + 32 * g + 16 * hh);
            const uint32_t qv[4] = {q.x, q.y, q.z, q.w};
            uint32_t lo[8], hi[8];  // bf16x2 words: weights 2e, 2e+1 of the 16 low / high
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t v = qv[e];
                // bytes 4e..4e+3: nibbles as exact floats
                float ql[4], qh[4];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    ql[b] = static_cast<float>((v >> (8 * b)) & 0xFu);
                    qh[b] = static_cast<float>((v >> (8 * b + 4)) & 0xFu);
                }
                lo[2 * e] = pack_bf16(fmaf(dl, ql[0], -ml), fmaf(dl, ql[1], -ml));
                lo[2 * e + 1] = pack_bf16(fmaf(dl, ql[2], -ml), fmaf(dl, ql[3], -ml));
                hi[2 * e] = pack_bf16(fmaf(dh, qh[0], -mh), fmaf(dh, qh[1], -mh));
                hi[2 * e + 1] = pack_bf16(fmaf(dh, qh[2], -mh), fmaf(dh, qh[3], -mh));
            }
            // low nibbles: k = 64g + 16hh + 0..15 -> chunks 8g + 2hh, +1
            // high nibbles: k = 64g + 32 + 16hh + 0..15 -> chunks 8g + 4 + 2hh, +1
            const int jl = 8 * g + 2 * hh, jh = 8 * g + 4 + 2 * hh;
            *reinterpret_cast<uint4*>(opA + op_off(t, jl)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4*>(opA + op_off(t, jl + 1)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
            *reinterpret_cast<uint4*>(opA + op_off(t, jh)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(opA + op_off(t, jh + 1)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_q4k_tc_kernel(const uint8_t* __restrict__ W, const float* __restrict__ X, float* __restrict__ Y, int M,
                       int64_t N, int64_t K, unsigned* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem);       // [2]
    uint64_t* raw_empty = raw_full + 2;                            // [2]
    uint64_t* op_full = raw_full + 4;
    uint64_t* op_empty = raw_full + 5;
    uint64_t* acc_full = raw_full + 6;
    uint64_t* acc_empty = raw_full + 7;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 128);
    uint8_t* opA = smem + kOpA0;
    uint8_t* opB = smem + kOpB0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = static_cast<int>(K / 256);
    const int64_t pitch = static_cast<int64_t>(nb) * kBlockBytes;
    const int64_t ntiles = (N + kTileRows - 1) / kTileRows;
    const int64_t U = ntiles * nb;
    const int64_t u_begin = U * blockIdx.x / gridDim.x;
    const int64_t u_end = U * (blockIdx.x + 1) / gridDim.x;
    const int nmma = M <= 16 ? 16 : 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 4);
        }
        mbar_init(op_full, 4);
        mbar_init(op_empty, 1);
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        fence_mbar_init();
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ---------------- producer
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        for (int64_t u = u_begin; u < u_end; ++u) {
            const int64_t i = u - u_begin;
            const int s = static_cast<int>(i & 1);
            if (i >= 2) mbar_wait_bounded(&raw_empty[s], static_cast<uint32_t>(((i >> 1) - 1) & 1), status);
            const int64_t tile = u / nb;
            const int kb = static_cast<int>(u % nb);
            const int64_t row0 = tile * kTileRows;
            const int rows = static_cast<int>(min64(kTileRows, N - row0));
            uint8_t* raw = smem + kRaw0 + s * kRawStage;
            if (lane == 0) mbar_arrive_expect_tx(&raw_full[s], rows * kBlockBytes + M * 1024);
            __syncwarp();
            const uint8_t* src = W + row0 * pitch + static_cast<int64_t>(kb) * kBlockBytes;
            for (int r = lane; r < rows; r += 32)
                bulk_g2s(raw + r * kBlockBytes, src + r * pitch, kBlockBytes, &raw_full[s], pol_w);
            for (int m = lane; m < M; m += 32)
                bulk_g2s(raw + kRawW + m * 1024, X + m * K + static_cast<int64_t>(kb) * 256, 1024, &raw_full[s],
                         pol_x);
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer
        const uint32_t idesc = instr_desc(kTileRows, nmma);
        const uint32_t a0 = smem_u32(opA), b0 = smem_u32(opB);
        int64_t seg = 0;
        for (int64_t u = u_begin; u < u_end; ++u) {
            const int64_t i = u - u_begin;
            const int kb = static_cast<int>(u % nb);
            const bool first = (u == u_begin) || kb == 0;
            const bool last = (u == u_end - 1) || kb == nb - 1;
            mbar_wait_bounded(op_full, static_cast<uint32_t>(i & 1), status);
            if (first && seg > 0) mbar_wait_bounded(acc_empty, static_cast<uint32_t>((seg - 1) & 1), status);
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int ks = 0; ks < 16; ++ks) {
                    const uint64_t ad = smem_desc(a0 + 256 * ks, 128, 4096);
                    const uint64_t bd = smem_desc(b0 + 256 * ks, 128, 4096);
                    mma_bf16(tmem, ad, bd, idesc, (first && ks == 0) ? 0u : 1u);
                }
                mma_commit(op_empty);
                if (last) mma_commit(acc_full);
            }
            __syncwarp();
            if (last) ++seg;
        }
        // the last segment's accumulator must be drained before TMEM is freed
        if (seg > 0) mbar_wait_bounded(acc_empty, static_cast<uint32_t>((seg - 1) & 1), status);
    } else {
        // ---------------- dequant + epilogue (warps 0-3, thread t = tile row t)
        const int t = threadIdx.x;
        int64_t seg = 0;
        for (int64_t u = u_begin; u < u_end; ++u) {
            const int64_t i = u - u_begin;
            const int s = static_cast<int>(i & 1);
            const int64_t tile = u / nb;
            const int kb = static_cast<int>(u % nb);
            const bool last = (u == u_end - 1) || kb == nb - 1;
            const int64_t row0 = tile * kTileRows;
            const int rows = static_cast<int>(min64(kTileRows, N - row0));
            const uint8_t* raw = smem + kRaw0 + s * kRawStage;
            mbar_wait_bounded(&raw_full[s], static_cast<uint32_t>((i >> 1) & 1), status);
            if (i >= 1) mbar_wait_bounded(op_empty, static_cast<uint32_t>((i - 1) & 1), status);
            if (t < rows) dequant_row(raw + t * kBlockBytes, opA, t);
            // X slice -> bf16 operand: chunk c = (token m, k chunk j)
            const float* xr = reinterpret_cast<const float*>(raw + kRawW);
            for (int c = t; c < M * 32; c += 128) {
                const int m = c >> 5, j = c & 31;
                const float4 a = *reinterpret_cast<const float4*>(xr + m * 256 + 8 * j);
                const float4 b = *reinterpret_cast<const float4*>(xr + m * 256 + 8 * j + 4);
                *reinterpret_cast<uint4*>(opB + op_off(m, j)) =
                    make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
            }
            fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
            __syncwarp();
            if (lane == 0) {
                arrive(&raw_empty[s]);
                arrive(op_full);
            }
            if (last) {
                mbar_wait_bounded(acc_full, static_cast<uint32_t>(seg & 1), status);
                tc_fence_after();
                float v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16), v);
                const int64_t row = row0 + t;
                if (t < rows) {
#pragma unroll
                    for (int m = 0; m < 32; ++m)
                        if (m < M) atomicAdd(&Y[m * N + row], v[m]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive(acc_empty);
                ++seg;
            }
        }
    }
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace tc

int launch_gemm_q4k_tc(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t s,
                       unsigned* status) {
    if (M < 16 || M > 32) return QG_EINVAL;
    static bool attr_done[64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ECUDA;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(tc::gemm_q4k_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc::kSmemTotal) != cudaSuccess)
            return QG_ECUDA;
        attr_done[dev] = true;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return QG_ECUDA;
    if (cudaMemsetAsync(Y, 0, static_cast<size_t>(M) * N * sizeof(float), s) != cudaSuccess) return QG_ECUDA;
    const int64_t units = ((N + tc::kTileRows - 1) / tc::kTileRows) * (K / 256);
    const int grid = static_cast<int>(std::min<int64_t>(units, sms));
    tc::gemm_q4k_tc_kernel<<<grid, tc::kThreads, tc::kSmemTotal, s>>>(W, X, Y, M, N, K, status);
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

}  // namespace qg
