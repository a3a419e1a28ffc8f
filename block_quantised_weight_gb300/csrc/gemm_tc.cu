// Batched Q4_K and IQ3 GEMM on the tcgen05 tensor cores.
//
//   Y[m][n] = sum_k w[n][k] * X[m][k]
//
// Two kernels, one CTA layout.  W rows sit on the MMA's M=128 side, tokens
// on its N=16/32 side (tcgen05.mma kind::f16, bf16 x bf16, fp32
// accumulation in tensor memory).
//   qg_gemm_tc_kernel (Q4_K, 16 <= M <= 32): a 128-row tile of W is
//     dequantised (page 1 "Rewriting picoLM in Python", dequantize_q4_K:
//     (d*sc)*q - dmin*mn) exactly in fp32 and rounded once to bf16 (to
//     nearest even); X is rounded to bf16 likewise.
//   qg_gemm_tc_x_kernel<Q4K, XP, MT> (Q4_K from 5 to 15 tokens, IQ3 from 5
//     tokens): each weight's small integer (Q4_K q - c, IQ3 the signed grid
//     byte) enters the MMA exactly and the sub-block factors are applied
//     after it (see there); x in XP bf16 parts (XP = 3 up to 10 tokens per
//     launch: exact products, the fp32 bar; XP = 1 from 16 tokens).
//
// CTA roles (320 threads):
//   warps 0-7  dequantise W into tensor memory and X into shared memory:
//              warps 0-3 the first 128 k of each unit, warps 4-7 the second
//              (thread = tile row = TMEM lane); then read the sums back
//              (tcgen05.ld, warp w reads TMEM lanes 32 (w mod 4) ..): in
//              qg_gemm_tc_kernel warps 0-3 drain the accumulator into Y per
//              segment, in the factored kernel each half's warps take their
//              sub-blocks' sums every unit;
//   warp 8     producer: one 2D tensor-map TMA per unit for the 128 rows x
//              block column of W (Q4_K: 144 bytes; IQ3: the 112 bytes from
//              the block's offset rounded down to 16, the block starting
//              0..14 bytes in) and one for the x slice (fp32), into a ring of
//              raw stages;
//   warp 9     allocates tensor memory; lane 0 issues the MMAs and commits
//              them to mbarriers.
// Work: units (tile, k-block) in row-major order, split evenly over the grid
// (stream-K); a CTA's run over one tile is a "segment" whose partial sums are
// added into Y (zeroed first) with fp32 atomics.  Each unit is dequantised
// in two halves of 128 k, in parallel.  The MMA takes its W operand (A, 128
// rows x 16 k per instruction) from tensor memory, written with tcgen05.st,
// and x (B) from shared memory.  Both are double-buffered per half, and so
// is the accumulator, so the dequantisation of one unit overlaps the MMAs
// of the one before, and a segment's drain the next segment's MMAs.
//
// Tensor memory (512 columns): A of half h, buffer b at columns 64 (2h + b)
// (row = lane, k pairs as bf16x2 per column, k ascending); the accumulators
// of qg_gemm_tc_kernel at 256 and 288 (D[row][token], fp32, 32 columns
// each), the factored kernel's sub-block sums at 256 + 128 h + 32 j.
//
// Exact Q4_K weights: with the fp16 magic h = 1024 + q, one fp16 FMA gives
// h*sc - 1024*sc = q*sc exactly (at most 945: the fused product is rounded
// once and the result is representable); a mixed f16 x f16 + f32 FMA then
// gives d*(q*sc) - dmin*mn with a single rounding, the pages' fp32 value.
//
// x operand layout (K-major, 128-byte swizzle): for half h, buffer b, two
// 4 KB atoms (k 0-63 and 64-127 of the half) of 32 token rows x 128 bytes;
// the 16-byte chunk j of row r sits at position j ^ (r mod 8), so eight
// rows' chunks j fall in eight distinct bank groups.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "gemv_kernel.cuh"
#include "launch.h"
#include "tensor_map.h"

namespace qg {
namespace tc {

constexpr int kTileRows = 128;
constexpr int kBlockBytes = 144;
constexpr int kThreads = 320;  // 8 dequant warps, producer, MMA
constexpr int kRawW = kTileRows * kBlockBytes;     // 18432: TMA box 144 x 128 (IQ3: 112 x 128, x after 18432 too)
constexpr int kIQ3Box = 112;
constexpr int kMaxRaw = 6;                          // raw stages (W box + the unit's x, M KB)
// Shared memory: barriers, the four x stages, (factored kernel) the IQ3
// tables or the Q4_K x sums, and the raw ring at the end: as many stages of
// kRawW + M * 1024 bytes as fit.
constexpr int kB0 = 1024;
constexpr int kBStage = 2 * 32 * 128;               // 8192: two 64-k atoms of 32 token rows
constexpr int kRaw0Q4K = kB0 + 4 * kBStage;         // 33792
constexpr int kSmemMax = 232448;                     // 227 KB per CTA
__host__ __device__ constexpr int raw_stage_bytes(int M) { return kRawW + M * 1024; }
constexpr int kTmemCols = 512;
constexpr uint32_t kTmA = 0;                        // A of half h, buffer b at kTmA + 64 (2h + b)
constexpr uint32_t kTmD = 256;                      // accumulator p at kTmD + 32 p
constexpr uint32_t kSBO = 8 * 128;                  // 8-row group stride in an x atom

// smem descriptor for tcgen05.mma, K-major with the 128-byte swizzle: start
// address, leading byte offset (unused by this layout: 16), stride byte
// offset between 8-row groups, descriptor version 1, base offset 0 (every
// atom starts on a 1024-byte boundary), swizzle mode 2 (128 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // version
    d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
    return d;
}

// instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t instr_desc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// D (+)= A B^T with A (128 rows x 16 k, bf16) in tensor memory at tmem_a.
__device__ __forceinline__ void mma_bf16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(tmem_d), "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
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

// 32 32-bit columns of this warp's 32 TMEM lanes (lane = thread), from registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&w)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
          "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
          "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
          "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Offset of the 16-byte chunk (token row m, k chunk j < 16 of the half) in an
// x stage: atom j / 8, row m at 128 m, chunk position (j mod 8) ^ (m mod 8).
__device__ __forceinline__ uint32_t x_off(int m, int j) {
    return static_cast<uint32_t>((j >> 3) * 4096 + m * 128 + (((j & 7) ^ (m & 7)) << 4));
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// fp32 d*qs + c, with d the fp16 in the low half of dh and qs one half of qp.
__device__ __forceinline__ float mfma_lo(uint32_t dh, uint32_t qp, float c) {
    float r;
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %3;\n\t}" : "=f"(r) : "r"(dh), "r"(qp), "f"(c));
    return r;
}
__device__ __forceinline__ float mfma_hi(uint32_t dh, uint32_t qp, float c) {
    float r;
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b1, %3;\n\t}" : "=f"(r) : "r"(dh), "r"(qp), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t half2_bits(float a) {
    const __half2 h = __floats2half2_rn(a, a);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Thread t: half `half` (k 128*half .. +127) of the W tile row t -> 64 bf16
// pairs in this thread's TMEM lane, columns ta .. ta + 63 (column c: k 2c, 2c+1).
__device__ __forceinline__ void dequant_half(const uint8_t* blk, uint32_t ta, int half) {
    const uint4 h = *reinterpret_cast<const uint4*>(blk);
    const uint32_t dbits = h.x & 0xFFFFu;
    const float dmin = h2f(h.x >> 16);
    uint32_t sc03, mn03, sc47, mn47;
    q4k_scale_min_words(h.y, h.z, h.w, sc03, mn03, sc47, mn47);
    const uint32_t scw = half == 0 ? sc03 : sc47, mnw = half == 0 ? mn03 : mn47;
#pragma unroll
    for (int gg = 0; gg < 2; ++gg) {
        const int g = 2 * half + gg;
        uint32_t w[32];  // k 64gg .. 64gg + 63 of the half: 8 chunks of 4 columns
        const float sl = byte_f(scw, 2 * gg), sh = byte_f(scw, 2 * gg + 1);
        const float ml = -(dmin * byte_f(mnw, 2 * gg)), mh = -(dmin * byte_f(mnw, 2 * gg + 1));
        // (1024+q)*sl - 1024*sl = q*sl; (1024+16q)*(sh/16) - 64*sh = q*sh (all exact in fp16)
        const uint32_t SL = half2_bits(sl), NL = half2_bits(-1024.f * sl);
        const uint32_t SH = half2_bits(sh * 0.0625f), NH = half2_bits(-64.f * sh);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint4 q = *reinterpret_cast<const uint4*>(blk + 16 + 32 * g + 16 * hh);
            const uint32_t qv[4] = {q.x, q.y, q.z, q.w};
            uint32_t lo[8], hi[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t v = qv[e], v8 = v >> 8;
                const uint32_t A = hfma2_u32((v & 0x000F000Fu) | 0x64006400u, SL, NL);   // q*sl, bytes 0,2
                const uint32_t C = hfma2_u32((v8 & 0x000F000Fu) | 0x64006400u, SL, NL);  // bytes 1,3
                const uint32_t B = hfma2_u32((v & 0x00F000F0u) | 0x64006400u, SH, NH);   // q*sh, bytes 0,2
                const uint32_t D = hfma2_u32((v8 & 0x00F000F0u) | 0x64006400u, SH, NH);  // bytes 1,3
                lo[2 * e] = pack_bf16(mfma_lo(dbits, A, ml), mfma_lo(dbits, C, ml));
                lo[2 * e + 1] = pack_bf16(mfma_hi(dbits, A, ml), mfma_hi(dbits, C, ml));
                hi[2 * e] = pack_bf16(mfma_lo(dbits, B, mh), mfma_lo(dbits, D, mh));
                hi[2 * e + 1] = pack_bf16(mfma_hi(dbits, B, mh), mfma_hi(dbits, D, mh));
            }
            // low nibbles: k' = 16hh + 0..15 (chunks 2hh, 2hh+1 of the 64); high: k' + 32
            const int jl = 2 * hh, jh = 4 + 2 * hh;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                w[4 * jl + e] = lo[e];
                w[4 * jl + 4 + e] = lo[4 + e];
                w[4 * jh + e] = hi[e];
                w[4 * jh + 4 + e] = hi[4 + e];
            }
        }
        tmem_st32(ta + 32 * gg, w);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    qg_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const uint8_t* __restrict__ grid, float* __restrict__ Y, int M, int64_t N, int64_t K, int nraw,
                   unsigned* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem);  // [kMaxRaw]
    uint64_t* raw_empty = raw_full + kMaxRaw;                 // [kMaxRaw]
    uint64_t* op_full = raw_full + 2 * kMaxRaw;               // [half][buffer]
    uint64_t* op_empty = op_full + 4;                         // [half][buffer]
    uint64_t* acc_full = op_full + 8;                         // [2]
    uint64_t* acc_empty = op_full + 10;                       // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
    const int raw0 = kRaw0Q4K;
    const int rstage = raw_stage_bytes(M);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = static_cast<int>(K / 256);
    const int64_t ntiles = (N + kTileRows - 1) / kTileRows;
    const int64_t U = ntiles * nb;
    const int64_t u_begin = U * blockIdx.x / gridDim.x;
    const int64_t u_end = U * (blockIdx.x + 1) / gridDim.x;
    const int nmma = M <= 16 ? 16 : 32;
    // the swizzled x stages need a 1024-byte aligned base (all threads see the
    // same address: the CTA leaves before any barrier or TMEM use)
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(status, kStatusBounds);
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < nraw; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 8);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&op_full[i], 4);
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        fence_mbar_init();
    }
    // x stages: token rows past M stay zero (the MMA reads 16 or 32 rows)
    for (int i = threadIdx.x; i < 4 * kBStage / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + kB0)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == 9) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ---------------- producer (one thread issues the tensor copies)
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            const uint32_t bytes = kTileRows * kBlockBytes + M * 1024;
            // (stage, phase, tile, k-block) kept incrementally: a 64-bit
            // division per unit costs a good fraction of a unit's time
            int s = 0;
            uint32_t round = 0;  // completed passes over the raw ring
            int64_t tile = u_begin / nb;
            int kb = static_cast<int>(u_begin % nb);
            for (int64_t u = u_begin; u < u_end; ++u) {
                if (u - u_begin >= nraw) mbar_wait_bounded(&raw_empty[s], (round - 1) & 1u, status);
                uint8_t* raw = smem + raw0 + s * rstage;
                mbar_arrive_expect_tx(&raw_full[s], bytes);
                tma_load_2d(raw, &tmW, kb * kBlockBytes, static_cast<int>(tile * kTileRows), &raw_full[s], pol_w);
                tma_load_2d(raw + kRawW, &tmX, kb * 256, 0, &raw_full[s], pol_x);
                if (++s == nraw) {
                    s = 0;
                    ++round;
                }
                if (++kb == nb) {
                    kb = 0;
                    ++tile;
                }
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ---------------- MMA issuer
        const uint32_t idesc = instr_desc(kTileRows, nmma);
        int64_t seg = 0;
        int kb = static_cast<int>(u_begin % nb);  // advanced at the end of each unit (no division per unit)
        for (int64_t u = u_begin; u < u_end; ++u, kb = kb + 1 == nb ? 0 : kb + 1) {
            const int64_t i = u - u_begin;
            const int b = static_cast<int>(i & 1);
            const bool first = (u == u_begin) || kb == 0;
            const bool last = (u == u_end - 1) || kb == nb - 1;
            const uint32_t td = tmem + kTmD + 32u * static_cast<uint32_t>(seg & 1);
            // both halves, then the unit's 16 MMAs in one straight run (a
            // branch between two MMAs doubles their issue cost)
            mbar_wait_bounded(&op_full[b], static_cast<uint32_t>((i >> 1) & 1), status);
            mbar_wait_bounded(&op_full[2 + b], static_cast<uint32_t>((i >> 1) & 1), status);
            if (first && seg >= 2)  // segment seg - 2 drained from this accumulator
                mbar_wait_bounded(&acc_empty[seg & 1], static_cast<uint32_t>(((seg >> 1) - 1) & 1), status);
            tc_fence_after();
            if (lane == 0) {
                const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t ta = tmem + kTmA + 64u * static_cast<uint32_t>(2 * h + b);
                    const uint32_t b0 = smem_u32(smem + kB0 + (2 * h + b) * kBStage);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {  // k 16 ks .. +15 of the half
                        const uint64_t bd = smem_desc_sw128(b0 + 4096 * (ks >> 2) + 32 * (ks & 3), kSBO);
                        mma_bf16_ta(td, ta + 8 * ks, bd, idesc, (h == 0 && ks == 0) ? acc0 : 1u);
                    }
                }
                mma_commit(&op_empty[b]);
                mma_commit(&op_empty[2 + b]);
                if (last) mma_commit(&acc_full[seg & 1]);
            }
            __syncwarp();
            if (last) ++seg;
        }
        // the last segments' accumulators must be drained before TMEM is freed
        for (int64_t q = seg >= 2 ? seg - 2 : 0; q < seg; ++q)
            mbar_wait_bounded(&acc_empty[q & 1], static_cast<uint32_t>((q >> 1) & 1), status);
    } else {
        // ---------------- dequant (warps 0-7) + epilogue (warps 0-3)
        const int half = warp >> 2;         // which 128 k of the unit
        const int t = threadIdx.x & 127;    // tile row = TMEM lane
        const int hw = warp & 3;            // TMEM lanes 32 hw .. 32 hw + 31
        const uint32_t tl = static_cast<uint32_t>(32 * hw) << 16;
        int64_t seg = 0;
        // (raw stage, its phase, tile, k-block) kept incrementally
        int s = 0;
        uint32_t rphase = 0;
        int64_t tile = u_begin / nb;
        int kb = static_cast<int>(u_begin % nb);
        for (int64_t u = u_begin; u < u_end; ++u) {
            const int64_t i = u - u_begin;
            const bool last = (u == u_end - 1) || kb == nb - 1;
            const int64_t row0 = tile * kTileRows;
            const int rows = static_cast<int>(min64(kTileRows, N - row0));
            const uint8_t* raw = smem + raw0 + s * rstage;
            const float* xr = reinterpret_cast<const float*>(raw + kRawW);
            const int b = static_cast<int>(i & 1);
            mbar_wait_bounded(&raw_full[s], rphase, status);
            // buffer b of this half was last read by the MMAs of unit i - 2
            if (i >= 2) mbar_wait_bounded(&op_empty[2 * half + b], static_cast<uint32_t>(((i >> 1) - 1) & 1), status);
            tc_fence_after();
            const uint32_t ta = tmem + tl + kTmA + 64u * static_cast<uint32_t>(2 * half + b);
            dequant_half(raw + t * kBlockBytes, ta, half);
            // x -> bf16 chunks (token m = c / 16, k chunk j = c mod 16 of the
            // half): a quarter warp takes one token's 8 consecutive chunks,
            // stored to 8 distinct bank groups; two-way loads
            {
                uint8_t* xs = smem + kB0 + (2 * half + b) * kBStage;
                for (int c = t; c < M * 16; c += 128) {
                    const int m = c >> 4, j = c & 15;
                    const float4 a = *reinterpret_cast<const float4*>(xr + m * 256 + 128 * half + 8 * j);
                    const float4 q = *reinterpret_cast<const float4*>(xr + m * 256 + 128 * half + 8 * j + 4);
                    *reinterpret_cast<uint4*>(xs + x_off(m, j)) = make_uint4(
                        pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(q.x, q.y), pack_bf16(q.z, q.w));
                }
            }
            tmem_wait_st();            // W in tensor memory
            fence_proxy_async_smem();  // x: generic-proxy stores -> visible to the tensor core
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                arrive(&op_full[2 * half + b]);
                arrive(&raw_empty[s]);
            }
            if (last && half == 0) {
                mbar_wait_bounded(&acc_full[seg & 1], static_cast<uint32_t>((seg >> 1) & 1), status);
                tc_fence_after();
                float v[32];
                tmem_ld32(tmem + tl + kTmD + 32u * static_cast<uint32_t>(seg & 1), v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive(&acc_empty[seg & 1]);
                if (t < rows) {
                    const int64_t row = row0 + t;
#pragma unroll
                    for (int m = 0; m < 32; ++m)
                        if (m < M) atomicAdd(&Y[m * N + row], v[m]);
                }
            }
            if (last) ++seg;
            if (++s == nraw) {
                s = 0;
                rphase ^= 1u;
            }
            if (++kb == nb) {
                kb = 0;
                ++tile;
            }
        }
    }
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}



// ------------------------------------ sub-block factors after the MMA
// Both formats write each weight as a small integer times a per-sub-block
// factor, and the MMA takes the integers, which bf16 holds exactly:
//   IQ3 (page 4 "iq3_pack.py", decode): w = d*(0.5+code)*0.5 * grid*0.5 *
//     sign = f_j * (+-g), g a grid byte, f_j = d*(0.5+code)*0.25;
//   Q4_K (page 1 "Rewriting picoLM in Python", dequantize_q4_K): w =
//     a*q - b with a = d*sc, b = dmin*mn of sub-block j; with the offset c
//     of q4k_offset (the integer nearest b/a) w = a*(q - c) - r, r = b - a*c,
//     and every term of a*sum((q-c)*x) - r*sum(x) is at most twice |w*x| of
//     its weight, so cancelling weights keep their accuracy.
// x enters as XP bf16 parts: XP = 3 splits each x exactly (x = hi + mid +
// lo, each part rounding the remainder of the one before), so every product
// is exact and only the fp32 sums round; XP = 1 rounds x to bf16.  Each
// (row, sub-block, token part) accumulates in its own TMEM column; the
// dequantising warps then add f_j * S (IQ3) or a_j * S - r_j * X_j (Q4_K; S
// the sum of the parts, X_j the sub-block's sum of x as the MMA saw it)
// into registers, a unit behind the MMAs.
// IQ3 grid in 16 copies: a half warp's 8-byte gathers (lane L reads copy
// L mod 16) fall in 16 distinct bank pairs whatever the grid rows.
constexpr int kGridX0 = kB0 + 4 * kBStage;       // 33792: IQ3 grid rows as two bf16 pairs, 16 copies (32 KB)
constexpr int kSignX0 = kGridX0 + 32768;         // 66560: IQ3 sign words, 8 copies (4 KB)
constexpr int kRaw0X3 = kSignX0 + 4096;          // 70656: IQ3 raw ring
constexpr int kXSum0 = kB0 + 4 * kBStage;        // 33792: Q4_K x sums [half][3 slots][4 sub-blocks][32 tokens]
constexpr int kRaw0XQ = kXSum0 + 2 * 3 * 4 * 32 * 4;  // 36864: Q4_K raw ring
constexpr uint32_t kTmDX = 256;                  // D of half h at 256 + 128 h, sub-block j at + 32 j

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// MT: the tokens a launch may carry (XP * MT <= 32 columns of D per
// sub-block), a compile-time bound so that the per-unit sums touch only
// those columns.
template <bool Q4K, int XP, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    qg_gemm_tc_x_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        const uint8_t* __restrict__ grid, float* __restrict__ Y, int M, int64_t N, int64_t K,
                        int nraw, unsigned* status) {
    static_assert(XP == 1 || XP == 3, "x parts");
    static_assert(XP * MT <= 32 && MT % 2 == 0, "tokens per launch");
    constexpr int kRaw0 = Q4K ? kRaw0XQ : kRaw0X3;
    constexpr int kBox = Q4K ? kBlockBytes : kIQ3Box;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem);  // [kMaxRaw]
    uint64_t* raw_empty = raw_full + kMaxRaw;                 // [kMaxRaw]
    uint64_t* op_full = raw_full + 2 * kMaxRaw;               // [half][buffer]
    uint64_t* op_empty = op_full + 4;                         // [half][buffer]
    uint64_t* d_full = op_full + 8;                           // [half]
    uint64_t* d_empty = op_full + 10;                         // [half]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
    const int rstage = raw_stage_bytes(M);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = static_cast<int>(K / 256);
    const int64_t ntiles = (N + kTileRows - 1) / kTileRows;
    const int64_t U = ntiles * nb;
    const int64_t u_begin = U * blockIdx.x / gridDim.x;
    const int64_t u_end = U * (blockIdx.x + 1) / gridDim.x;
    const int ncol = XP * M <= 16 ? 16 : 32;
    // the swizzled x stages need a 1024-byte aligned base (all threads see the
    // same address: the CTA leaves before any barrier or TMEM use)
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(status, kStatusBounds);
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < nraw; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 8);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&op_full[i], 4);
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], 4);
        }
        fence_mbar_init();
    }
    // x stages: token rows past XP * M stay zero (the MMA reads 16 or 32 rows)
    for (int i = threadIdx.x; i < 4 * kBStage / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + kB0)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if constexpr (!Q4K) {
        // grid row r as bf16 pairs (bytes 0,1) (bytes 2,3), 16 copies: row r of copy c at 8 (16 r + c) bytes
        uint2* g2 = reinterpret_cast<uint2*>(smem + kGridX0);
        for (int i = threadIdx.x; i < 256 * 16; i += kThreads) {
            const uint8_t* gr = grid + (i >> 4) * 4;
            g2[i] = make_uint2(pack_bf16(gr[0], gr[1]), pack_bf16(gr[2], gr[3]));
        }
        // signs of each 7-bit field: the seven stored ones and their parity
        // (page 4, decode), sign k at bit 15 - k/2 (k even) or 31 - k/2 (odd)
        uint32_t* sg = reinterpret_cast<uint32_t*>(smem + kSignX0);
        for (int i = threadIdx.x; i < 8 * 128; i += kThreads) {  // i = 8 * s7 + copy
            const uint32_t s7 = static_cast<uint32_t>(i) >> 3;
            const uint32_t s8 = s7 | ((__popc(s7) & 1u) << 7);
            uint32_t t = 0;
            for (int pr = 0; pr < 4; ++pr)
                t |= (((s8 >> (2 * pr)) & 1u) << (15 - pr)) | (((s8 >> (2 * pr + 1)) & 1u) << (31 - pr));
            sg[i] = t;
        }
    }
    if (warp == 9) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ---------------- producer (one thread issues the tensor copies)
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            const uint32_t bytes = kTileRows * kBox + M * 1024;
            int s = 0;
            uint32_t round = 0;  // completed passes over the raw ring
            int64_t tile = u_begin / nb;
            int kb = static_cast<int>(u_begin % nb);
            for (int64_t u = u_begin; u < u_end; ++u) {
                if (u - u_begin >= nraw) mbar_wait_bounded(&raw_empty[s], (round - 1) & 1u, status);
                uint8_t* raw = smem + kRaw0 + s * rstage;
                mbar_arrive_expect_tx(&raw_full[s], bytes);
                const int bx = Q4K ? kb * kBlockBytes : (kb * 98) & ~15;  // x * 1 byte: 16-byte aligned
                tma_load_2d(raw, &tmW, bx, static_cast<int>(tile * kTileRows), &raw_full[s], pol_w);
                tma_load_2d(raw + kRawW, &tmX, kb * 256, 0, &raw_full[s], pol_x);
                if (++s == nraw) {
                    s = 0;
                    ++round;
                }
                if (++kb == nb) {
                    kb = 0;
                    ++tile;
                }
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ---------------- MMA issuer: per unit both halves, 16 MMAs in one run
        const uint32_t idesc = instr_desc(kTileRows, ncol);
        for (int64_t i = 0; i < u_end - u_begin; ++i) {
            const int b = static_cast<int>(i & 1);
            mbar_wait_bounded(&op_full[b], static_cast<uint32_t>((i >> 1) & 1), status);
            mbar_wait_bounded(&op_full[2 + b], static_cast<uint32_t>((i >> 1) & 1), status);
            if (i >= 1) {  // the previous unit's sums read out of D
                mbar_wait_bounded(&d_empty[0], static_cast<uint32_t>((i - 1) & 1), status);
                mbar_wait_bounded(&d_empty[1], static_cast<uint32_t>((i - 1) & 1), status);
            }
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t ta = tmem + kTmA + 64u * static_cast<uint32_t>(2 * h + b);
                    const uint32_t td = tmem + kTmDX + 128u * static_cast<uint32_t>(h);
                    const uint32_t b0 = smem_u32(smem + kB0 + (2 * h + b) * kBStage);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {  // sub-block ks / 2 of the half: two MMAs of 16 k
                        const uint64_t bd = smem_desc_sw128(b0 + 4096 * (ks >> 2) + 32 * (ks & 3), kSBO);
                        mma_bf16_ta(td + 32 * (ks >> 1), ta + 8 * ks, bd, idesc, static_cast<uint32_t>(ks & 1));
                    }
                }
                mma_commit(&op_empty[b]);
                mma_commit(&op_empty[2 + b]);
                mma_commit(&d_full[0]);
                mma_commit(&d_full[1]);
            }
            __syncwarp();
        }
    } else {
        // ---------------- dequant (warps 0-7: half = warp / 4, thread = tile row = TMEM lane)
        const int half = warp >> 2;
        const int t = threadIdx.x & 127;
        const uint32_t tl = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        float* xsum = reinterpret_cast<float*>(smem + kXSum0) + half * (3 * 4 * 32);  // Q4_K: [slot][sub-block][token]
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        float fp[4] = {0.f, 0.f, 0.f, 0.f};  // the previous unit's sub-block factors (IQ3 f, Q4_K a)
        float rp[4] = {0.f, 0.f, 0.f, 0.f};  // and Q4_K offsets' remainders r
        int64_t prow0 = 0;
        int prows = 0;
        bool plast = false;
        // the previous unit's sums into acc; at a segment's end acc goes into Y
        auto drain = [&](int64_t ip) {
            mbar_wait_bounded(&d_full[half], static_cast<uint32_t>(ip & 1), status);
            tc_fence_after();
            const float* xs = xsum + static_cast<int>(ip % 3) * (4 * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v[32];
                tmem_ld32(tmem + tl + kTmDX + 128u * static_cast<uint32_t>(half) + 32u * j, v);
                if (j == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive(&d_empty[half]);
                }
#pragma unroll
                for (int m = 0; m < MT; m += 2) {
                    const float s0 = XP == 1 ? v[m] : v[3 * m] + (v[3 * m + 1] + v[3 * m + 2]);
                    const float s1 = XP == 1 ? v[m + 1] : v[3 * m + 3] + (v[3 * m + 4] + v[3 * m + 5]);
                    acc[m] = fmaf(fp[j], s0, acc[m]);
                    acc[m + 1] = fmaf(fp[j], s1, acc[m + 1]);
                    if constexpr (Q4K) {
                        const float2 xx = *reinterpret_cast<const float2*>(xs + j * 32 + m);
                        acc[m] = fmaf(-rp[j], xx.x, acc[m]);
                        acc[m + 1] = fmaf(-rp[j], xx.y, acc[m + 1]);
                    }
                }
            }
            if (plast) {
                if (t < prows) {
                    const int64_t row = prow0 + t;
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < M) atomicAdd(&Y[m * N + row], acc[m]);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = 0.f;
            }
        };
        int s = 0;
        uint32_t rphase = 0;
        int64_t tile = u_begin / nb;
        int kb = static_cast<int>(u_begin % nb);
        for (int64_t u = u_begin; u < u_end; ++u) {
            const int64_t i = u - u_begin;
            const int b = static_cast<int>(i & 1);
            const bool last = (u == u_end - 1) || kb == nb - 1;
            const int64_t row0 = tile * kTileRows;
            const int rows = static_cast<int>(min64(kTileRows, N - row0));
            const uint8_t* raw = smem + kRaw0 + s * rstage;
            const float* xr = reinterpret_cast<const float*>(raw + kRawW);
            mbar_wait_bounded(&raw_full[s], rphase, status);
            // buffer b of this half was last read by the MMAs of unit i - 2
            if (i >= 2) mbar_wait_bounded(&op_empty[2 * half + b], static_cast<uint32_t>(((i >> 1) - 1) & 1), status);
            tc_fence_after();
            const uint32_t ta = tmem + tl + kTmA + 64u * static_cast<uint32_t>(2 * half + b);
            float f[4], r[4];
            if constexpr (Q4K) {
                // row t's sub-blocks 4 half .. 4 half + 3: a = d*sc, b = dmin*mn, offset c, r = b - a*c
                const uint8_t* blk = raw + t * kBlockBytes;
                const uint4 hd = *reinterpret_cast<const uint4*>(blk);
                const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
                uint32_t sc03, mn03, sc47, mn47;
                q4k_scale_min_words(hd.y, hd.z, hd.w, sc03, mn03, sc47, mn47);
                const uint32_t scw = half == 0 ? sc03 : sc47, mnw = half == 0 ? mn03 : mn47;
                uint32_t cneg[4];  // bf16 pairs of 128 + c
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a = d * byte_f(scw, j), bb = dmin * byte_f(mnw, j);
                    const float c = q4k_offset(a, bb);
                    f[j] = a;
                    r[j] = bb - a * c;
                    cneg[j] = (0x4300u | static_cast<uint32_t>(c)) * 0x10001u;
                }
                // q - c as bf16: a byte permute puts q next to 0x43 (bf16 128 + q),
                // and one bf16x2 subtraction takes 128 + c off, both exact
#pragma unroll
                for (int gg = 0; gg < 2; ++gg) {  // sub-blocks 2gg (low nibbles) and 2gg + 1 (high)
                    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 64 * half + 32 * gg);
                    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 16 + 64 * half + 32 * gg + 16);
                    const uint32_t qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                    uint32_t w[32];  // k 64gg .. 64gg + 63 of the half
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t L = qv[e] & 0x0F0F0F0Fu, H = (qv[e] >> 4) & 0x0F0F0F0Fu;
                        w[2 * e] = bf16x2_sub(prmt(L, 0x43434343u, 0x4140u), cneg[2 * gg]);
                        w[2 * e + 1] = bf16x2_sub(prmt(L, 0x43434343u, 0x4342u), cneg[2 * gg]);
                        w[16 + 2 * e] = bf16x2_sub(prmt(H, 0x43434343u, 0x4140u), cneg[2 * gg + 1]);
                        w[16 + 2 * e + 1] = bf16x2_sub(prmt(H, 0x43434343u, 0x4342u), cneg[2 * gg + 1]);
                    }
                    tmem_st32(ta + 32 * gg, w);
                }
            } else {
                const uint2* g2 = reinterpret_cast<const uint2*>(smem + kGridX0);
                const uint32_t* sgn = reinterpret_cast<const uint32_t*>(smem + kSignX0);
                uint32_t vi[8], vs[4], dbits;
                switch (kb & 7) {  // the block's offset in its box: (98 * kb) mod 16
#define QG_TC_IQ3X(C) \
    case C: iq3_load_half<FmtIQ3T, C>(raw + t * kIQ3Box, half, vi, vs, dbits); break;
                    QG_TC_IQ3X(0) QG_TC_IQ3X(1) QG_TC_IQ3X(2) QG_TC_IQ3X(3)
                    QG_TC_IQ3X(4) QG_TC_IQ3X(5) QG_TC_IQ3X(6) QG_TC_IQ3X(7)
#undef QG_TC_IQ3X
                }
                const float d = h2f(dbits);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    f[j] = d * (static_cast<float>(vs[j] >> 28) + 0.5f) * 0.25f;
                    r[j] = 0.f;
                }
                // the signed grid bytes as bf16, sub-block j at columns 16 j .. 16 j + 15
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    uint32_t w[32];
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int j = 2 * jp + jj;
                        const uint32_t sw = vs[j];
#pragma unroll
                        for (int l = 0; l < 4; ++l) {
                            const uint32_t T = sgn[8 * ((sw >> (7 * l)) & 0x7Fu) + (t & 7)];
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const int pi = 8 * j + 2 * l + hf;  // index byte within the half
                                const uint32_t idx = (vi[pi >> 2] >> (8 * (pi & 3))) & 0xFFu;
                                const uint2 g = g2[16 * idx + (t & 15)];
                                w[16 * jj + 4 * l + 2 * hf] = g.x ^ ((T << (2 * hf)) & 0x80008000u);
                                w[16 * jj + 4 * l + 2 * hf + 1] = g.y ^ ((T << (2 * hf + 1)) & 0x80008000u);
                            }
                        }
                    }
                    tmem_st32(ta + 32 * jp, w);
                }
            }
            // x -> XP bf16 parts, part p of token m in row XP m + p; Q4_K also
            // the sums of x as the MMA sees it per (token, sub-block): the four
            // chunks of a sub-block are four consecutive lanes
            {
                uint8_t* xs = smem + kB0 + (2 * half + b) * kBStage;
                float* xsw = xsum + static_cast<int>(i % 3) * (4 * 32);
                for (int n = 0; n < (M * 16 + 127) / 128; ++n) {  // the same trip count in every lane
                    const int c = t + 128 * n, m = c >> 4, j = c & 15;
                    float part = 0.f;
                    if (m < M) {
                        const float4 a = *reinterpret_cast<const float4*>(xr + m * 256 + 128 * half + 8 * j);
                        const float4 q = *reinterpret_cast<const float4*>(xr + m * 256 + 128 * half + 8 * j + 4);
                        float v[8] = {a.x, a.y, a.z, a.w, q.x, q.y, q.z, q.w};
                        if constexpr (Q4K && XP == 3) part = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
#pragma unroll
                        for (int p = 0; p < XP; ++p) {
                            uint32_t w4[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                w4[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
                                const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xFFFF0000u);
                                if constexpr (Q4K && XP == 1) part += lo + hi;
                                // the remainder is exact in fp32 (Sterbenz)
                                v[2 * e] -= lo;
                                v[2 * e + 1] -= hi;
                            }
                            *reinterpret_cast<uint4*>(xs + x_off(XP * m + p, j)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                    if constexpr (Q4K) {
                        part += __shfl_xor_sync(0xffffffffu, part, 1);
                        part += __shfl_xor_sync(0xffffffffu, part, 2);
                        if (m < M && (j & 3) == 0) xsw[(j >> 2) * 32 + m] = part;
                    }
                }
            }
            tmem_wait_st();            // W in tensor memory
            fence_proxy_async_smem();  // x: generic-proxy stores -> visible to the tensor core
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                arrive(&op_full[2 * half + b]);
                arrive(&raw_empty[s]);
            }
            // Q4_K: this unit's x sums for the whole half (three slots: a thread
            // rewrites slot (i + 1) mod 3 only after every thread of the half
            // passed this barrier, that is, left the drain of unit i - 2)
            if constexpr (Q4K) named_barrier_sync<128>(1 + half);
            if (i >= 1) drain(i - 1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                fp[j] = f[j];
                rp[j] = r[j];
            }
            plast = last;
            prow0 = row0;
            prows = rows;
            if (++s == nraw) {
                s = 0;
                rphase ^= 1u;
            }
            if (++kb == nb) {
                kb = 0;
                ++tile;
            }
        }
        if (u_end > u_begin) drain(u_end - u_begin - 1);
    }
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace tc


namespace {

// Both formats: W viewed as [N rows][pitch bytes] with a box of one block
// column (Q4_K 144 bytes; IQ3 112 bytes) x 128 rows; X [M][K] fp32 with a
// box of 256 k x M tokens.  FMT 0: Q4_K with weights rounded to bf16
// (qg_gemm_tc_kernel, 16 <= M <= 32); FMT 1 / 2: IQ3 / Q4_K with the
// sub-block factors after the MMA and x in XP bf16 parts (XP * M <= 32).
template <int FMT, int XP>
int launch_tc(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
              cudaStream_t s, unsigned* status) {
    constexpr bool IQ3 = FMT == 1;
    if (FMT == 0 ? (M < 16 || M > 32) : (M < 1 || XP * M > 32)) return QG_EINVAL;
    static std::atomic<bool> attr_done[2][64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return qg::cuda_fail(cudaGetLastError());
    // the factored kernel with the smaller token bound that holds M
    constexpr int kMT0 = XP == 3 ? 8 : 16, kMT1 = 32 / XP / 2 * 2;
    const bool small = M <= kMT0;
    auto kern = FMT == 0 ? tc::qg_gemm_tc_kernel
                : small  ? tc::qg_gemm_tc_x_kernel<FMT == 2, XP, kMT0>
                         : tc::qg_gemm_tc_x_kernel<FMT == 2, XP, kMT1>;
    std::atomic<bool>& attr = attr_done[small ? 0 : 1][dev];
    // as many raw stages as fit (the x part of a stage is M KB)
    const int raw0 = FMT == 0 ? tc::kRaw0Q4K : IQ3 ? tc::kRaw0X3 : tc::kRaw0XQ;
    const int nraw = std::min(tc::kMaxRaw, (tc::kSmemMax - raw0) / tc::raw_stage_bytes(M));
    if (nraw < 2) return QG_EINVAL;
    const int smem = raw0 + nraw * tc::raw_stage_bytes(M);
    if (!attr.load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemMax) != cudaSuccess)
            return qg::cuda_fail(cudaGetLastError());
        attr.store(true, std::memory_order_release);
    }
    auto encode = tensor_map_encoder();
    if (!encode) return qg::cuda_fail(cudaGetLastError());
    const uint64_t pitch = static_cast<uint64_t>(K / 256) * (IQ3 ? 98 : tc::kBlockBytes);
    CUtensorMap tmW, tmX;
    if (!encode_byte_rows(&tmW, W, pitch, static_cast<uint64_t>(N), IQ3 ? tc::kIQ3Box : tc::kBlockBytes,
                          tc::kTileRows))
        return qg::cuda_fail(cudaGetLastError());
    {
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(K) * 4};
        const cuuint32_t box[2] = {256, static_cast<cuuint32_t>(M)};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(X), gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return qg::cuda_fail(cudaGetLastError());
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return qg::cuda_fail(cudaGetLastError());
    if (cudaMemsetAsync(Y, 0, static_cast<size_t>(M) * N * sizeof(float), s) != cudaSuccess) return qg::cuda_fail(cudaGetLastError());
    const int64_t units = ((N + tc::kTileRows - 1) / tc::kTileRows) * (K / 256);
    const int gridx = static_cast<int>(std::min<int64_t>(units, sms));
    kern<<<gridx, tc::kThreads, smem, s>>>(tmW, tmX, grid, Y, M, N, K, nraw, status);
    return launch_status();
}

}  // namespace

int launch_gemm_q4k_tc(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t s,
                       unsigned* status) {
    return launch_tc<0, 1>(W, nullptr, X, Y, M, N, K, s, status);
}

// IQ3 needs 16-byte aligned rows (K/256 a multiple of 8) for its tensor map.
int launch_gemm_iq3_tc(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                       cudaStream_t s, unsigned* status) {
    if ((K / 256) % 8 != 0) return QG_EINVAL;
    return launch_tc<1, 1>(W, grid, X, Y, M, N, K, s, status);
}

// IQ3, 1 <= M <= 10, x in three bf16 parts: every product exact, fp32 sums.
int launch_gemm_iq3_tc3(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                        cudaStream_t s, unsigned* status) {
    if ((K / 256) % 8 != 0) return QG_EINVAL;
    return launch_tc<1, 3>(W, grid, X, Y, M, N, K, s, status);
}

// Q4_K, 1 <= M <= 10, x in three bf16 parts: every product exact, fp32 sums,
// the offset factoring of the FMA path.
int launch_gemm_q4k_tc3(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t s,
                        unsigned* status) {
    return launch_tc<2, 3>(W, nullptr, X, Y, M, N, K, s, status);
}

}  // namespace qg
