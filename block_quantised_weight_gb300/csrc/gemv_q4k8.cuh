// Q4_K GEMV for 5 to 8 tokens in one pass over W (fp32 FMA path).
//
// The 4-token kernel of gemv_kernel.cuh needs about 168 registers a thread,
// the most a 9-warp CTA gets (three warps share one scheduler's 16K
// registers), so more tokens would take a second pass over W and decode
// every weight twice.  This kernel has 8 warps and no producer warp, so a
// thread may hold up to 255 registers: warp w streams block column w of
// every 8-column unit through a ring of its own (lane 0 issues the weight
// box and the tokens' x slices, the lanes consume them), and the 8 warps
// meet only at the end of a tile, to add their row sums.  The decode is the
// one of the other Q4_K kernels (q4k_stage_x, q4k_half2: page 1 "Rewriting
// picoLM in Python", dequantize_q4_K, with the exact offset factoring), so
// its results follow the same arithmetic.
#pragma once
#include "launch_common.cuh"

namespace qg {
namespace q8 {

constexpr int kWarps = kCols;       // one warp per block column of a unit
constexpr int kBox = kRows * 144;   // a column's weight box: 32 rows x 144 B
constexpr int kMaxS = 4;            // ring stages per warp (upper bound)

struct Layout8 {
    int sx, red, ring, stage, total;
};
// barriers [kWarps][kMaxS] at 0; per-warp sub-block sums of x; row sums of
// two tile parities; the rings, warp w's S stages of (box, MT x slices).
__host__ __device__ inline Layout8 layout8(int MT, int S) {
    Layout8 L;
    L.sx = 8 * kWarps * kMaxS;
    L.red = L.sx + align_up(kWarps * MT * 8 * 4, 128);
    L.ring = L.red + align_up(2 * kWarps * MT * kRows * 4, 128);
    L.stage = kBox + MT * 1024;
    L.total = L.ring + kWarps * S * L.stage;
    return L;
}

template <int MT>
__global__ void __launch_bounds__(kWarps * 32, 1)
    qg_gemv8_kernel(const __grid_constant__ Group G, const __grid_constant__ TMaps T, const float* __restrict__ X,
                    int M, int64_t K, int S, unsigned* status, int flags) {
    static_assert(MT >= 1 && MT <= 8, "tokens per launch");
    extern __shared__ __align__(128) uint8_t smem[];
    const Layout8 L = layout8(MT, S);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = static_cast<int>(K / 256);
    const int64_t ntiles = G.tile0[G.count];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem) + warp * kMaxS;
    float* sxp = reinterpret_cast<float*>(smem + L.sx) + warp * MT * 8;
    float* red = reinterpret_cast<float*>(smem + L.red);
    uint8_t* ring = smem + L.ring + warp * S * L.stage;

    grid_launch_dependents();
    const bool prefetch = (flags & kFlagPrefetchWeights) != 0;
    if (!prefetch) grid_dependency_wait();
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane < G.count) prefetch_tensormap(&T.m[lane]);
    __syncwarp();

    // this warp's units: the CTA's tiles blockIdx.x, + gridDim.x, ..., and
    // in each the chunks c whose column c*8 + warp exists
    struct Pos {
        int64_t tile;
        int c;
    };
    auto advance = [&](Pos& p) {
        if (++p.c * kWarps + warp >= nb) {
            p.c = 0;
            p.tile += gridDim.x;
        }
    };
    const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
    auto post = [&](const Pos& p, int s, bool do_w, bool do_x, bool expect) {
        const int gi = group_find(G, p.tile);
        const int64_t row0 = (p.tile - G.tile0[gi]) * kRows;
        const int col = p.c * kWarps + warp;
        uint8_t* st = ring + s * L.stage;
        if (expect && lane == 0) mbar_arrive_expect_tx(&full[s], kBox + M * 1024);
        __syncwarp();
        // rows past N arrive as zeros and count toward the transaction bytes
        if (do_w && lane == 0) tma_load_2d(st, &T.m[gi], col * 144, static_cast<int>(row0), &full[s], pol_w);
        if (do_x && lane < M)
            bulk_g2s(st + kBox + lane * 1024, X + lane * K + static_cast<int64_t>(col) * 256, 1024, &full[s], pol_x);
    };

    const bool has_units = warp < nb && static_cast<int64_t>(blockIdx.x) < ntiles;
    Pos pp{static_cast<int64_t>(blockIdx.x), 0};  // next unit to post
    int ps = 0;                                      // its slot
    if (has_units) {
        // the first S units: weights at once (before the dependency wait
        // when prefetching), x after it
        Pos q = pp;
        int n = 0;
        for (; n < S && q.tile < ntiles; ++n, advance(q)) post(q, n, true, !prefetch, true);
        if (prefetch) {
            grid_dependency_wait();
            Pos r = pp;
            for (int i = 0; i < n; ++i, advance(r)) post(r, i, false, true, false);
        }
        pp = q;
        ps = n % S;
    } else if (prefetch) {
        grid_dependency_wait();
    }

    float acc2[2][MT], ss[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc2[0][m] = acc2[1][m] = ss[m] = 0.f;
    int s = 0;
    uint32_t phase = 0;
    int64_t tile_count = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tile_count) {
        const int gi = group_find(G, tile);
        const int64_t row0 = (tile - G.tile0[gi]) * kRows, Ni = G.N[gi];
        const int rows = static_cast<int>(min64(kRows, Ni - row0));
        if (warp < nb) {
            for (int c = 0; c * kWarps + warp < nb; ++c) {
                mbar_wait_bounded(&full[s], phase, status);
                uint8_t* st = ring + s * L.stage;
                float* xb = reinterpret_cast<float*>(st + kBox);
                float e2[MT];
                const bool rescaled = q4k_stage_x<MT, 128>(xb, 256, nullptr, 0, sxp, ss, e2, M, lane);
                __syncwarp();
                // two rows per lane (lane&15 and +16), half lane>>4 of the block
                const uint8_t* blk = st + (lane & 15) * 144;
                if (rescaled)  // rare; the same in every lane
                    q4k_half2<MT, 128, true>(blk, 16 * 144, lane >> 4, xb, 256, sxp, M, e2, acc2);
                else
                    q4k_half2<MT, 128, false>(blk, 16 * 144, lane >> 4, xb, 256, sxp, M, e2, acc2);
                fence_proxy_async_smem();  // x was written in place: order it before the slot's next copy
                __syncwarp();              // every lane is done with the slot
                if (pp.tile < ntiles) {
                    post(pp, ps, true, true, true);
                    advance(pp);
                    if (++ps == S) ps = 0;
                }
                if (++s == S) {
                    s = 0;
                    phase ^= 1u;
                }
            }
        }
        // the 8 column warps' row sums -> Y (every warp takes part, with or
        // without columns in this tile)
        float* rb = red + (tile_count & 1) * (kWarps * MT * kRows);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float s0 = acc2[0][m] + __shfl_xor_sync(0xffffffffu, acc2[0][m], 16);
            const float s1 = acc2[1][m] + __shfl_xor_sync(0xffffffffu, acc2[1][m], 16);
            rb[(warp * MT + m) * kRows + lane] = lane < 16 ? s0 : s1;
            acc2[0][m] = acc2[1][m] = 0.f;
        }
        named_barrier_sync<kWarps * 32>(1);
        for (int t = threadIdx.x; t < MT * kRows; t += kWarps * 32) {
            const int m = t / kRows, rr = t % kRows;
            if (m < M && rr < rows) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) sum += rb[(w * MT + m) * kRows + rr];
                G.Y[gi][m * Ni + row0 + rr] = sum;
            }
        }
    }
}

}  // namespace q8

// Launch qg_gemv8_kernel over `count` matrices sharing X (token offset m0
// applied to X; Y[i] + m0 * N[i] here), M <= 8 tokens: one CTA per SM, as
// many ring stages per warp as fit (at least two).
inline int launch_gemv8(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, int m0,
                        const float* X, int M, int64_t K, cudaStream_t s, unsigned* status, int dev,
                        unsigned flags) {
    static std::atomic<bool> attr_done[64];
    constexpr int MT = 8;
    int S = q8::kMaxS;
    while (S > 2 && q8::layout8(MT, S).total > kSmemPerCTA) --S;
    const q8::Layout8 L = q8::layout8(MT, S);
    if (L.total > kSmemPerCTA) return QG_EINVAL;
    auto kern = q8::qg_gemv8_kernel<MT>;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) != cudaSuccess)
            return qg::cuda_fail(cudaGetLastError());
        attr_done[dev].store(true, std::memory_order_release);
    }
    Group G = {};
    G.count = count;
    G.tile0[0] = 0;
    for (int i = 0; i < count; ++i) {
        G.W[i] = W[i];
        G.Y[i] = Y[i] + static_cast<int64_t>(m0) * N[i];
        G.N[i] = N[i];
        G.tile0[i + 1] = G.tile0[i] + (N[i] + kRows - 1) / kRows;
    }
    TMaps T = {};
    const uint64_t pitch = static_cast<uint64_t>(K / 256) * 144;
    for (int i = 0; i < count; ++i)
        if (!encode_byte_rows(&T.m[i], W[i], pitch, static_cast<uint64_t>(N[i]), 144, kRows))
            return qg::cuda_fail(cudaGetLastError());
    const int sms = sm_count(dev);
    if (sms <= 0) return qg::cuda_fail(cudaGetLastError());
    const int grid = static_cast<int>(std::min<int64_t>(G.tile0[count], sms));
    const int kflags = (flags & QG_PREFETCH_WEIGHTS) ? kFlagPrefetchWeights : 0;
    if (!(flags & QG_PREFETCH_WEIGHTS)) {
        kern<<<grid, q8::kWarps * 32, L.total, s>>>(G, T, X, M, K, S, status, kflags);
        return launch_status();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(q8::kWarps * 32);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, G, T, X, M, K, S, status, kflags) != cudaSuccess)
        return qg::cuda_fail(cudaGetLastError());
    return launch_status();
}

}  // namespace qg
