// Host-only probe for tests/test_layout_host.py: prints, for every
// configuration the tcgen05 launchers can choose (format, x parts, tokens),
// the shared-memory and tensor-memory layout that launch_tc derives from
// gemm_tc.cu's constants (same stage rule), one JSON object per line.  The
// kernels are compiled with the file but never launched.
#include <cstdio>

#include "gemm_tc.cu"

using namespace qg;

// fmt 0: qg_gemm_tc_kernel (Q4_K, bf16 weights); 1 / 2: the factored kernel
// for IQ3 / Q4_K with x in xp bf16 parts
static void emit(int fmt, int xp, int M) {
    const int raw0 = fmt == 0 ? tc::kRaw0Q4K : fmt == 1 ? tc::kRaw0X3 : tc::kRaw0XQ;
    const int stage = tc::raw_stage_bytes(M);
    const int nraw = std::min(tc::kMaxRaw, (tc::kSmemMax - raw0) / stage);
    // the end of what sits below the raw ring: x stages, then the IQ3 tables
    // or the Q4_K x sums
    const int below = fmt == 0 ? tc::kB0 + 4 * tc::kBStage
                      : fmt == 1 ? tc::kSignX0 + 4096
                                 : tc::kXSum0 + 2 * 3 * 4 * 32 * 4;
    const int barriers = fmt == 0 ? 2 * tc::kMaxRaw + 4 + 4 + 2 + 2 : 2 * tc::kMaxRaw + 4 + 4 + 2 + 2;
    const int ncol = fmt == 0 ? (M <= 16 ? 16 : 32) : (xp * M <= 16 ? 16 : 32);
    // TMEM: A buffers at 0..255; accumulators (fmt 0) at 256 + 32 p, p < 2;
    // sub-block sums (factored) at 256 + 128 h + 32 j, j < 4, ncol wide
    const int tmem_end = fmt == 0 ? tc::kTmD + 32 * 2 : tc::kTmDX + 128 + 32 * 3 + ncol;
    std::printf(
        "{\"fmt\": %d, \"xp\": %d, \"M\": %d, \"raw0\": %d, \"stage\": %d, \"nraw\": %d, \"smem\": %d, "
        "\"smem_max\": %d, \"below\": %d, \"b0\": %d, \"b_stage\": %d, \"x_rows\": %d, \"ncol\": %d, "
        "\"barrier_bytes\": %d, \"tmem_slot\": %d, \"tmem_end\": %d, \"tmem_cols\": %d, \"box_bytes\": %d, "
        "\"raw_w\": %d, \"tile_rows\": %d}\n",
        fmt, xp, M, raw0, stage, nraw, raw0 + nraw * stage, tc::kSmemMax, below, tc::kB0, tc::kBStage, xp * M, ncol,
        8 * barriers, 512, tmem_end, tc::kTmemCols, fmt == 1 ? tc::kIQ3Box : tc::kBlockBytes, tc::kRawW,
        tc::kTileRows);
}

int main() {
    for (int M = 16; M <= 32; ++M) emit(0, 1, M);   // qgemm_q4k_batched from 16 tokens
    for (int M = 16; M <= 32; ++M) emit(1, 1, M);   // qgemm_iq3_batched from 16 tokens
    for (int M = 1; M <= 10; ++M) emit(1, 3, M);    // IQ3 groups of up to 10 tokens
    for (int M = 1; M <= 10; ++M) emit(2, 3, M);    // Q4_K groups of up to 10 tokens
    return 0;
}
