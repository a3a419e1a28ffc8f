// Host-only probe for tests/test_layout_host.py: prints, for every kernel
// configuration the GEMV launchers can choose, the shared-memory layout
// that launch_gemv derives (same budget and stage rule), one JSON object
// per line.  No kernel is instantiated or launched.
#include <cstdio>

#include "gemv_kernel.cuh"

using namespace qg;

template <class F>
static void emit(const char* fmt, int MT, int RG, int MINB, int fuse) {
    const int budget = std::min(kSmemPerCTA, kSmemPerSM / MINB - kSmemReserve);
    const Layout L1 = make_layout(F::kIQ3, MT, F::kXH, RG, 1, F::kRowStride, F::kCols, fuse, F::kWPC);
    const int fit = std::min(kMaxStages, (budget - L1.stage0) / L1.stage_bytes);
    const Layout L = make_layout(F::kIQ3, MT, F::kXH, RG, fit, F::kRowStride, F::kCols, fuse, F::kWPC);
    std::printf(
        "{\"fmt\": \"%s\", \"MT\": %d, \"RG\": %d, \"MINB\": %d, \"fuse\": %d, \"budget\": %d, \"stages\": %d, "
        "\"full\": %d, \"empty\": %d, \"sx\": %d, \"red\": %d, \"cred\": %d, \"ss\": %d, \"table\": %d, "
        "\"stage0\": %d, \"stage_bytes\": %d, \"xoff\": %d, \"aoff\": %d, \"total\": %d, "
        "\"block_bytes\": %d, \"box_bytes\": %d, \"tile_rows\": %d, \"cols\": %d, \"xh\": %d, \"x_box_bytes\": %u, "
        "\"max_stages\": %d, \"smem_per_cta\": %d, \"warps\": %d}\n",
        fmt, MT, RG, MINB, fuse, budget, fit, L.full, L.empty, L.sx, L.red, L.cred, L.ss, L.table, L.stage0,
        L.stage_bytes, L.xoff, L.aoff, L.total, F::kBytes, F::kBoxBytes, RG * kRows, F::kCols, F::kXH, kXBoxBytes,
        kMaxStages, kSmemPerCTA, RG * F::kCols * F::kWPC);
}

int main() {
    // Q4_K (launch_q4k.cuh): one token at 2 or 1 CTAs per SM, two tokens,
    // four tokens; each with the fused prologues
    for (int fuse = 0; fuse <= 2; ++fuse) {
        emit<FmtQ4KT>("q4k", 1, 1, 2, fuse);
        emit<FmtQ4KT>("q4k", 1, 1, 1, fuse);
        emit<FmtQ4KT>("q4k", 2, 1, fuse == 0 ? 2 : 1, fuse);
        emit<FmtQ4KT>("q4k", 4, 1, 1, fuse);
    }
    // the prologue kernels of one token at one CTA per SM: two warps per column
    emit<FmtQ4KT2>("q4k2", 1, 1, 1, 1);
    emit<FmtQ4KT2>("q4k2", 1, 1, 1, 2);
    // IQ3, both block orders (launch_iq3.cuh): one token over 64-row tiles,
    // 2 and 4 tokens over 32-row tiles
    emit<FmtIQ3T>("iq3", 1, 2, 1, 0);
    emit<FmtIQ3T>("iq3", 2, 1, 1, 0);
    emit<FmtIQ3T>("iq3", 4, 1, 1, 0);
    emit<FmtIQ3XXST>("iq3xxs", 1, 2, 1, 0);
    emit<FmtIQ3XXST>("iq3xxs", 2, 1, 1, 0);
    emit<FmtIQ3XXST>("iq3xxs", 4, 1, 1, 0);
    return 0;
}
