// A whole decode pass of Q4_K GEMVs in one persistent kernel.
//
// The pass is a list of stages; a stage is a group of up to four matrices
// that read the same X (page 1 "Rewriting picoLM in Python", model_forward:
// q/k/v read the attention-norm output, gate/up the FFN-norm output), and
// stage s+1 may read what stage s wrote.  One cooperative launch (all CTAs
// resident) walks every stage with the same producer/consumer pipeline as
// qg_gemv_kernel; between stages a grid-wide completion count replaces the
// kernel boundary:
//   * each CTA, after writing its last Y of stage s (named barrier among its
//     consumers, then __threadfence), adds 1 to sync[s];
//   * the producer streams the weights of stage s+1 as soon as ring slots are
//     free, but issues the x copies of stage s+1 only after sync[s] reaches
//     the grid size (bounded spin; acquire load, then a generic->async proxy
//     fence so the bulk copies see the stored values).
// Weights never wait for the previous stage; only the activations do.
// All CTAs are resident (cooperative launch), so the waits always end; they
// are bounded all the same and report QG_ETIMEOUT.
#include <algorithm>

#include "launch_common.cuh"

namespace qg {
namespace pass {

constexpr int kMaxStagesPass = QG_MAX_PASS_STAGES;

struct Stage {
    Group G;
    const float* X;
    int64_t K;
    int nb;
    int nchunks;
};
struct Plan {
    Stage st[kMaxStagesPass];
    int nstages;
};

__device__ __forceinline__ uint32_t ld_acquire(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_volatile(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *p >= target.  Returns false (timeout bit set) on expiry.
// Fails fast, without waiting, once this CTA has given up on an earlier
// count (gave_up) or once the status word carries a timeout that it did not
// carry when the kernel started (status0): a pass whose counts were reset
// under it (an overlapping call on the shared no-allocation scratch) would
// otherwise wait the full limit at every later stage.  Skipping a count wait
// only lets x be copied early; every copy still completes before use.
__device__ __forceinline__ bool wait_count(const unsigned* p, uint32_t target, unsigned* status, uint32_t status0,
                                           bool& gave_up) {
    if (ld_acquire(p) >= target) return true;
    if (gave_up) return false;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(64);
        if (ld_acquire(p) >= target) return true;
        if ((i & 15u) == 0) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
            if ((ld_volatile(status) & ~status0 & kStatusTimeout) != 0u) {  // someone else timed out meanwhile
                gave_up = true;
                return false;
            }
        }
    }
    atomicOr(status, kStatusTimeout);
    gave_up = true;
    return false;
}

// CTAs per SM: two for one and two tokens; a 4-token stage (32 rows of
// blocks plus 4 x 8 KB of x, 69 KB) needs one CTA per SM to keep two stages.
template <int MT>
constexpr int pass_ctas_per_sm() { return MT == 4 ? 1 : 2; }

template <int MT>
__global__ void __launch_bounds__(kCols * 32 + 32, pass_ctas_per_sm<MT>())
    qg_gemv_pass_kernel(const __grid_constant__ Plan P, int M, unsigned* sync, int stages, unsigned* status) {
    using F = FmtQ4K;
    constexpr int kWarps = kCols;  // one row group
    constexpr int kConsumerThreads = kWarps * 32;
    constexpr int kTileRows = kRows;
    extern __shared__ __align__(128) uint8_t smem[];
    const Layout L = make_layout(false, MT, F::kXH, 1, stages, F::kRowStride);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    float* sxw = reinterpret_cast<float*>(smem + L.sx);
    float* red = reinterpret_cast<float*>(smem + L.red);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kWarps) {
        // ---------------- producer warp
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        int s = 0;
        uint32_t round = 0;   // completed passes over the ring
        int64_t posted = 0;   // units posted so far (all stages)
        int def_s[kMaxStages], def_c[kMaxStages];
        const uint32_t status0 = ld_volatile(status);  // timeouts already reported before this launch
        bool gave_up = false;
        for (int si = 0; si < P.nstages; ++si) {
            const Stage& S = P.st[si];
            const int64_t pitch = static_cast<int64_t>(S.nb) * F::kBytes;
            const int64_t ntiles = S.G.tile0[S.G.count];
            bool deferring = si > 0;
            int ndef = 0;
            auto release_x = [&]() {
                if (lane == 0) wait_count(&sync[si - 1], gridDim.x, status, status0, gave_up);
                __syncwarp();
                asm volatile("fence.proxy.async.global;" ::: "memory");
                for (int k = 0; k < ndef; ++k) {
                    const int kc = min(kCols, S.nb - def_c[k] * kCols);
                    uint8_t* st = smem + L.stage0 + def_s[k] * L.stage_bytes;
                    if (lane < M)
                        bulk_g2s(st + L.xoff + lane * kCols * 1024,
                                 S.X + lane * S.K + static_cast<int64_t>(def_c[k]) * kCols * 256, kc * 1024,
                                 &full[def_s[k]], pol_x);
                }
                deferring = false;
                ndef = 0;
            };
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                const int gi = group_find(S.G, tile);
                const int64_t row0 = (tile - S.G.tile0[gi]) * kTileRows;
                const int rows = static_cast<int>(min64(kTileRows, S.G.N[gi] - row0));
                for (int c = 0; c < S.nchunks; ++c) {
                    if (posted >= stages) mbar_wait_bounded(&empty[s], (round - 1) & 1u, status);
                    const int kc = min(kCols, S.nb - c * kCols);
                    uint8_t* st = smem + L.stage0 + s * L.stage_bytes;
                    if (lane == 0) mbar_arrive_expect_tx(&full[s], rows * kc * F::kBytes + M * kc * 1024);
                    __syncwarp();
                    const uint8_t* src = S.G.W[gi] + row0 * pitch + static_cast<int64_t>(c) * kCols * F::kBytes;
                    for (int r = lane; r < rows; r += 32)
                        bulk_g2s(st + r * F::kRowStride, src + r * pitch, kc * F::kBytes, &full[s], pol_w);
                    if (deferring) {
                        def_s[ndef] = s;
                        def_c[ndef] = c;
                        ++ndef;
                        if (ndef == stages) release_x();
                    } else if (lane < M) {
                        bulk_g2s(st + L.xoff + lane * kCols * 1024, S.X + lane * S.K + static_cast<int64_t>(c) * kCols * 256,
                                 kc * 1024, &full[s], pol_x);
                    }
                    ++posted;
                    if (++s == stages) {
                        s = 0;
                        ++round;
                    }
                }
            }
            if (deferring && ndef > 0) release_x();
        }
        // nothing in flight is left unconsumed: consumers wait on every unit
    } else {
        // ---------------- consumer warps
        const int cw = warp;
        float acc[2][MT];  // rows (lane&15) and (lane&15)+16, half lane>>4 of each block
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[0][m] = acc[1][m] = 0.f;
        int s = 0;
        uint32_t phase = 0;
        int64_t tile_count = 0;
        for (int si = 0; si < P.nstages; ++si) {
            const Stage& S = P.st[si];
            const int64_t ntiles = S.G.tile0[S.G.count];
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                const int gi = group_find(S.G, tile);
                const int64_t row0 = (tile - S.G.tile0[gi]) * kTileRows;
                const int64_t Ni = S.G.N[gi];
                const int rows = static_cast<int>(min64(kTileRows, Ni - row0));
                for (int c = 0; c < S.nchunks; ++c) {
                    const int kc = min(kCols, S.nb - c * kCols);
                    const uint8_t* st = smem + L.stage0 + s * L.stage_bytes;
                    mbar_wait_bounded(&full[s], phase, status);
                    if (cw < kc) {
                        const float* xb = reinterpret_cast<const float*>(st + L.xoff) + cw * 256;
                        constexpr int64_t xstride = kCols * 256;
                        float* sxp = sxw + warp * MT * 8;
                        float ssq[MT], e2[MT];  // ssq unused: no prologue here
                        const bool rescaled =
                            q4k_stage_x<MT, 128>(const_cast<float*>(xb), xstride, nullptr, 0, sxp, ssq, e2, M, lane);
                        __syncwarp();
                        // two rows per lane, half a block each (same arithmetic as the
                        // single-launch GEMV; rows past the tile end are discarded)
                        const uint8_t* blk = st + (lane & 15) * F::kRowStride + cw * F::kBytes;
                        if (rescaled)
                            q4k_half2<MT, 128, true>(blk, 16 * F::kRowStride, lane >> 4, xb, xstride, sxp, M, e2, acc);
                        else
                            q4k_half2<MT, 128, false>(blk, 16 * F::kRowStride, lane >> 4, xb, xstride, sxp, M, e2, acc);
                        fence_proxy_async_smem();  // x was written: order it before the slot's next copy
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    if (c == S.nchunks - 1) {
                        float* rb = red + (tile_count & 1) * (kWarps * MT * kRows);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const float s0 = acc[0][m] + __shfl_xor_sync(0xffffffffu, acc[0][m], 16);
                            const float s1 = acc[1][m] + __shfl_xor_sync(0xffffffffu, acc[1][m], 16);
                            rb[(warp * MT + m) * kRows + lane] = lane < 16 ? s0 : s1;
                            acc[0][m] = acc[1][m] = 0.f;
                        }
                        named_barrier_sync<kConsumerThreads>(1);
                        for (int t = threadIdx.x; t < MT * kTileRows; t += kConsumerThreads) {
                            const int m = t / kTileRows, rr = t % kTileRows;
                            if ((MT == 1 || m < M) && rr < rows) {
                                float sum = 0.f;
#pragma unroll
                                for (int w = 0; w < kCols; ++w) sum += rb[(w * MT + m) * kRows + rr];
                                S.G.Y[gi][m * Ni + row0 + rr] = sum;
                            }
                        }
                        ++tile_count;
                    }
                    if (++s == stages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
            }
            // this CTA's part of stage si is written: publish it.  The barrier
            // orders every consumer's Y stores before thread 0's gpu-scope
            // fence, which releases them (cumulatively) ahead of the count; a
            // fence in each storing thread as well is not needed.
            named_barrier_sync<kConsumerThreads>(1);
            if (threadIdx.x == 0) {
                __threadfence();
                atomicAdd(&sync[si], 1u);
            }
        }
    }
}

}  // namespace pass

namespace {

template <int MT>
int launch_pass_t(const pass::Plan& plan, int M, unsigned* sync, cudaStream_t s, unsigned* status, int dev) {
    static std::atomic<bool> attr_done[64];
    static std::atomic<int> occ_cache[64];
    constexpr int kCtas = pass::pass_ctas_per_sm<MT>();
    const int budget = std::min(kSmemPerCTA, kSmemPerSM / kCtas - kSmemReserve);
    const Layout L1 = make_layout(false, MT, FmtQ4K::kXH, 1, 1, FmtQ4K::kRowStride);
    int stages = std::min(kMaxStages, (budget - L1.stage0) / L1.stage_bytes);
    if (stages < 2) return QG_EINVAL;
    const Layout L = make_layout(false, MT, FmtQ4K::kXH, 1, stages, FmtQ4K::kRowStride);
    auto kern = pass::qg_gemv_pass_kernel<MT>;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) != cudaSuccess)
            return qg::cuda_fail(cudaGetLastError());
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kCols * 32 + 32, L.total) != cudaSuccess ||
            occ < 1)
            return qg::cuda_fail(cudaGetLastError());
        occ_cache[dev].store(occ, std::memory_order_relaxed);
        attr_done[dev].store(true, std::memory_order_release);  // publishes occ_cache[dev]
    }
    const int sms = sm_count(dev);
    if (sms <= 0) return qg::cuda_fail(cudaGetLastError());
    const int grid = sms * std::min(occ_cache[dev].load(std::memory_order_relaxed), kCtas);
    if (cudaMemsetAsync(sync, 0, sizeof(unsigned) * plan.nstages, s) != cudaSuccess) return qg::cuda_fail(cudaGetLastError());
    void* args[] = {const_cast<pass::Plan*>(&plan), &M, &sync, &stages, &status};
    if (cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kCols * 32 + 32), args,
                                    L.total, s) != cudaSuccess)
        return qg::cuda_fail(cudaGetLastError());
    return launch_status();
}

}  // namespace

int launch_pass_q4k(const qg_stage* stages, int nstages, int M, unsigned* sync, cudaStream_t s, unsigned* status) {
    const int dev = current_device();
    if (dev < 0) return qg::cuda_fail(cudaGetLastError());
    thread_local pass::Plan plan;  // ~16 KB, kept off the stack; copied into the launch's parameters
    plan.nstages = nstages;
    for (int i = 0; i < nstages; ++i) {
        pass::Stage& S = plan.st[i];
        const qg_stage& q = stages[i];
        S.G = Group{};
        S.G.count = q.count;
        S.G.tile0[0] = 0;
        for (int j = 0; j < q.count; ++j) {
            S.G.W[j] = q.W[j];
            S.G.Y[j] = q.Y[j];
            S.G.N[j] = q.N[j];
            S.G.tile0[j + 1] = S.G.tile0[j] + (q.N[j] + kRows - 1) / kRows;
        }
        S.X = q.X;
        S.K = q.K;
        S.nb = static_cast<int>(q.K / 256);
        S.nchunks = (S.nb + kCols - 1) / kCols;
    }
    if (M == 1) return launch_pass_t<1>(plan, M, sync, s, status, dev);
    if (M == 2) return launch_pass_t<2>(plan, M, sync, s, status, dev);
    return launch_pass_t<4>(plan, M, sync, s, status, dev);
}

}  // namespace qg
