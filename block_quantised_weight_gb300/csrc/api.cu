// C-ABI entry points of libqgemv.so (declared in include/qgemv.h).
//
// Every argument is checked on the host before anything is launched; no
// exception crosses this boundary and nothing here aborts the process.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "gemv_kernel.cuh"
#include "launch.h"

namespace {

// Per-device status word: kernels OR qg::kStatus* bits into it.  Kernels get
// its device address (cudaGetSymbolAddress, cached per device), never the
// host-side symbol.
__device__ unsigned qg_status_word;
std::atomic<unsigned*> g_status_ptr[64];  // filled on first use; racing threads store the same value

unsigned* status_ptr() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    unsigned* p = g_status_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, qg_status_word) != cudaSuccess) return nullptr;
        p = static_cast<unsigned*>(a);
        g_status_ptr[dev].store(p, std::memory_order_relaxed);
    }
    return p;
}

}  // namespace

// Scratch of qgemv_q4k_pass_noalloc: its per-stage completion counts.  A
// fixed array in the library's own module, so that the entry point needs no
// allocation; every device that loads the library holds it until exit.  In
// host code `qg_noalloc_scratch` is a host-side stand-in for the symbol, not
// a device address: kernels get the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned qg_noalloc_scratch[QG_NOALLOC_SCRATCH_WORDS];
// A pass's plan holds QG_MAX_PASS_STAGES stages: the scratch never admits more.
static_assert(QG_NOALLOC_SCRATCH_WORDS <= QG_MAX_PASS_STAGES, "no-allocation scratch larger than a pass's plan");

namespace {

std::mutex g_noalloc_mu;
unsigned* g_noalloc_ptr[64];

// Set-up, once per device, with that device current: the device address of
// qg_noalloc_scratch.
int noalloc_scratch(unsigned** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return qg::cuda_fail(cudaGetLastError());
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, qg_noalloc_scratch) != cudaSuccess || !p) return qg::cuda_fail(cudaGetLastError());
        g_noalloc_ptr[dev] = static_cast<unsigned*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return QG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

// Shape checks shared by the GEMV entry points.  Sizes are bounded so that
// every byte count below fits comfortably in int64.
int check_gemv(const uint8_t* W, const uint8_t* grid, bool need_grid, const float* X, const float* Y, int M,
               int64_t N, int64_t K, int block_bytes) {
    if (!W || !X || !Y || (need_grid && !grid)) return QG_EINVAL;
    if (M < 1 || M > QG_MAX_M || N <= 0 || K <= 0 || K % 256 != 0) return QG_EINVAL;
    if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31)) return QG_EINVAL;
    if (!aligned16(W) || !aligned16(X) || !aligned16(Y) || (need_grid && !aligned16(grid))) return QG_EALIGN;
    const int64_t wbytes = N * (K / 256) * block_bytes;
    const int64_t ybytes = int64_t(M) * N * 4, xbytes = int64_t(M) * K * 4;
    if (overlap(Y, ybytes, W, wbytes) || overlap(Y, ybytes, X, xbytes) || (need_grid && overlap(Y, ybytes, grid, 1024)))
        return QG_EALIAS;
    return QG_OK;
}

int check_dequant(const uint8_t* W, const uint8_t* grid, bool need_grid, const float* out, int64_t N, int64_t K,
                  int block_bytes) {
    if (!W || !out || (need_grid && !grid)) return QG_EINVAL;
    if (N <= 0 || K <= 0 || K % 256 != 0 || N > (int64_t(1) << 31) || K > (int64_t(1) << 31)) return QG_EINVAL;
    if (N * (K / 256) > (int64_t(1) << 33)) return QG_EINVAL;
    if (!aligned16(W) || !aligned16(out) || (need_grid && !aligned16(grid))) return QG_EALIGN;
    if (overlap(out, N * K * 4, W, N * (K / 256) * block_bytes) || (need_grid && overlap(out, N * K * 4, grid, 1024)))
        return QG_EALIAS;
    return QG_OK;
}

// Test-only: an mbarrier nobody arrives on; the bounded wait must give up.
__global__ void qg_bounded_wait_probe(unsigned* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        qg::mbar_init(&bar, 1);
        qg::fence_mbar_init();
    }
    __syncthreads();
    qg::mbar_wait_bounded(&bar, 0, status, 20000000ull);  // 20 ms
}

}  // namespace

extern "C" {

int qgemv_q4k_ex(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, unsigned flags,
                 cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(QG_PREFETCH_WEIGHTS)) return QG_EINVAL;
    int rc = check_gemv(W, nullptr, false, X, Y, M, N, K, 144);
    if (rc != QG_OK) return rc;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    return qg::launch_gemv_q4k(W, X, Y, M, N, K, stream, st, flags);
}

int qgemv_q4k(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t stream) {
    return qgemv_q4k_ex(W, X, Y, M, N, K, 0u, stream);
}

int qgemv_iq3_ex(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                 unsigned flags, cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(QG_PREFETCH_WEIGHTS)) return QG_EINVAL;
    int rc = check_gemv(W, grid, true, X, Y, M, N, K, 98);
    if (rc != QG_OK) return rc;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    return qg::launch_gemv_iq3(W, grid, X, Y, M, N, K, stream, st, flags);
}

int qgemv_iq3(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
              cudaStream_t stream) {
    return qgemv_iq3_ex(W, grid, X, Y, M, N, K, 0u, stream);
}

int qgemv_iq3xxs_ex(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                    unsigned flags, cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(QG_PREFETCH_WEIGHTS)) return QG_EINVAL;
    int rc = check_gemv(W, grid, true, X, Y, M, N, K, 98);
    if (rc != QG_OK) return rc;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    return qg::launch_gemv_iq3xxs(W, grid, X, Y, M, N, K, stream, st, flags);
}

int qgemv_iq3xxs(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                 cudaStream_t stream) {
    return qgemv_iq3xxs_ex(W, grid, X, Y, M, N, K, 0u, stream);
}

static int64_t codebook_bytes(int format) {
    return format == QG_CB_IQ4_NL || format == QG_CB_IQ4_XS ? 16 : 2048;
}

int qgemv_codebook(int format, const uint8_t* W, const void* codebook, const float* X, float* Y, int M, int64_t N,
                   int64_t K, cudaStream_t stream) {
    if (format < QG_CB_IQ4_NL || format > QG_CB_IQ2_XXS || !codebook) return QG_EINVAL;
    const uint8_t* book = static_cast<const uint8_t*>(codebook);
    int rc = check_gemv(W, nullptr, false, X, Y, M, N, K, qg::cb_unit_bytes(format));
    if (rc != QG_OK) return rc;
    if (!aligned16(book)) return QG_EALIGN;
    if (overlap(Y, int64_t(M) * N * 4, book, codebook_bytes(format))) return QG_EALIAS;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    return qg::launch_gemv_cb(format, W, book, X, Y, M, N, K, stream, st);
}

int qdequant_codebook(int format, const uint8_t* W, const void* codebook, float* out, int64_t N, int64_t K,
                      cudaStream_t stream) {
    if (format < QG_CB_IQ4_NL || format > QG_CB_IQ2_XXS || !codebook) return QG_EINVAL;
    const uint8_t* book = static_cast<const uint8_t*>(codebook);
    int rc = check_dequant(W, nullptr, false, out, N, K, qg::cb_unit_bytes(format));
    if (rc != QG_OK) return rc;
    if (!aligned16(book)) return QG_EALIGN;
    if (overlap(out, N * K * 4, book, codebook_bytes(format))) return QG_EALIAS;
    return qg::launch_dequant_cb(format, W, book, out, N, K, stream);
}

// Group checks: every matrix as a single GEMV, plus no Y[i] overlapping any
// other matrix's W or Y.
static int check_group(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const uint8_t* grid,
                bool need_grid, const float* X, int M, int64_t K, int block_bytes) {
    if (!W || !Y || !N || count < 1 || count > QG_MAX_GROUP) return QG_EINVAL;
    for (int i = 0; i < count; ++i) {
        const int rc = check_gemv(W[i], grid, need_grid, X, Y[i], M, N[i], K, block_bytes);
        if (rc != QG_OK) return rc;
    }
    for (int i = 0; i < count; ++i)
        for (int j = 0; j < count; ++j) {
            if (i == j) continue;
            if (overlap(Y[i], int64_t(M) * N[i] * 4, W[j], N[j] * (K / 256) * block_bytes) ||
                overlap(Y[i], int64_t(M) * N[i] * 4, Y[j], int64_t(M) * N[j] * 4))
                return QG_EALIAS;
        }
    return QG_OK;
}

int qgemv_q4k_group(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const float* X, int M,
                    int64_t K, unsigned flags, cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(QG_PREFETCH_WEIGHTS)) return QG_EINVAL;
    int rc = check_group(W, Y, N, count, nullptr, false, X, M, K, 144);
    if (rc != QG_OK) return rc;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    return qg::launch_group_q4k(W, Y, N, count, X, M, K, stream, st, flags, nullptr);
}

// Fused calls: the group checks, then the prologue operands and residuals.
static int check_fuse(const qg_fuse* f, float* const* Y, const int64_t* N, int count, int M, int64_t K) {
    if (!f) return QG_OK;
    if (f->norm_weight && f->up) return QG_EINVAL;
    if ((f->norm_weight || f->up) && M > 4) return QG_EINVAL;
    if (f->norm_weight && !(f->norm_eps >= 0.f && f->norm_eps <= 3.0e38f)) return QG_EINVAL;
    if ((f->norm_weight && !aligned16(f->norm_weight)) || (f->up && !aligned16(f->up))) return QG_EALIGN;
    for (int i = 0; i < count; ++i) {
        const int64_t yb = int64_t(M) * N[i] * 4;
        if (f->residual[i] && !aligned16(f->residual[i])) return QG_EALIGN;
        if ((f->norm_weight && overlap(Y[i], yb, f->norm_weight, K * 4)) ||
            (f->up && overlap(Y[i], yb, f->up, int64_t(M) * K * 4)))
            return QG_EALIAS;
        for (int j = 0; j < count; ++j) {
            const float* r = f->residual[j];
            if (!r) continue;
            // a residual may be its own matrix's output, exactly; nothing else
            if (j == i ? (r != Y[i] && overlap(Y[i], yb, r, yb)) : overlap(Y[i], yb, r, int64_t(M) * N[j] * 4))
                return QG_EALIAS;
        }
    }
    return QG_OK;
}

static qg::Fuse to_fuse(const qg_fuse* f) {
    qg::Fuse z = {};
    if (f) {
        z.g = f->norm_weight;
        z.eps = f->norm_eps;
        z.up = f->up;
        for (int i = 0; i < QG_MAX_GROUP; ++i) z.R[i] = f->residual[i];
    }
    return z;
}

int qgemv_q4k_fused_group(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const float* X,
                          int M, int64_t K, const qg_fuse* fuse, unsigned flags, cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(QG_PREFETCH_WEIGHTS)) return QG_EINVAL;
    int rc = check_group(W, Y, N, count, nullptr, false, X, M, K, 144);
    if (rc != QG_OK) return rc;
    rc = check_fuse(fuse, Y, N, count, M, K);
    if (rc != QG_OK) return rc;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    const qg::Fuse z = to_fuse(fuse);
    return qg::launch_group_q4k_fused(W, Y, N, count, X, M, K, stream, st, flags, z);
}

int qgemv_q4k_fused(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, const qg_fuse* fuse,
                    unsigned flags, cudaStream_t stream) {
    if (fuse)
        for (int i = 1; i < QG_MAX_GROUP; ++i)
            if (fuse->residual[i]) return QG_EINVAL;
    return qgemv_q4k_fused_group(&W, &Y, &N, 1, X, M, K, fuse, flags, stream);
}

int qgemv_iq3_group(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const uint8_t* grid,
                    const float* X, int M, int64_t K, unsigned flags, cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(QG_PREFETCH_WEIGHTS)) return QG_EINVAL;
    int rc = check_group(W, Y, N, count, grid, true, X, M, K, 98);
    if (rc != QG_OK) return rc;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    return qg::launch_group_iq3(W, Y, N, count, grid, X, M, K, stream, st, flags);
}

int qgemv_q4k_pass(const qg_stage* stages, int nstages, int M, unsigned* sync, cudaStream_t stream) {
    if (!stages || !sync || nstages < 1 || nstages > QG_MAX_PASS_STAGES || M < 1 || M > 4) return QG_EINVAL;
    if (reinterpret_cast<uintptr_t>(sync) & 3u) return QG_EALIGN;
    for (int i = 0; i < nstages; ++i) {
        const qg_stage& q = stages[i];
        const int rc = check_group(q.W, const_cast<float* const*>(q.Y), q.N, q.count, nullptr, false, q.X, M, q.K, 144);
        if (rc != QG_OK) return rc;
        for (int j = 0; j < q.count; ++j)
            if (overlap(sync, 4 * int64_t(nstages), q.Y[j], int64_t(M) * q.N[j] * 4) ||
                overlap(sync, 4 * int64_t(nstages), q.W[j], q.N[j] * (q.K / 256) * 144))
                return QG_EALIAS;
    }
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    return qg::launch_pass_q4k(stages, nstages, M, sync, stream, st);
}

int qgemv_q4k_pass_noalloc(const qg_stage* stages, int nstages, int M, cudaStream_t stream) {
    if (!stages || nstages < 1 || M < 1 || M > 4) return QG_EINVAL;
    if (nstages > QG_NOALLOC_SCRATCH_WORDS) return QG_ESCRATCH;
    if (nstages > QG_MAX_PASS_STAGES) return QG_EINVAL;  // unreachable while the static_assert holds
    for (int i = 0; i < nstages; ++i) {
        const qg_stage& q = stages[i];
        const int rc = check_group(q.W, const_cast<float* const*>(q.Y), q.N, q.count, nullptr, false, q.X, M, q.K, 144);
        if (rc != QG_OK) return rc;
    }
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    unsigned* scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc != QG_OK) return rc;
    // launch_pass_q4k zeroes scratch[0, nstages) on the stream, then launches.
    return qg::launch_pass_q4k(stages, nstages, M, scratch, stream, st);
}

int qgemm_q4k_batched(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t stream) {
    int rc = check_gemv(W, nullptr, false, X, Y, M, N, K, 144);
    if (rc != QG_OK) return rc;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    if (M < 16) return qg::launch_gemv_q4k(W, X, Y, M, N, K, stream, st, 0u);
    return qg::launch_gemm_q4k_tc(W, X, Y, M, N, K, stream, st);
}

int qgemm_iq3_batched(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                      cudaStream_t stream) {
    int rc = check_gemv(W, grid, true, X, Y, M, N, K, 98);
    if (rc != QG_OK) return rc;
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    if (M < 16 || (K / 256) % 8 != 0) return qg::launch_gemv_iq3(W, grid, X, Y, M, N, K, stream, st, 0u);
    return qg::launch_gemm_iq3_tc(W, grid, X, Y, M, N, K, stream, st);
}

int qdequant_q4k(const uint8_t* W, float* out, int64_t N, int64_t K, cudaStream_t stream) {
    int rc = check_dequant(W, nullptr, false, out, N, K, 144);
    if (rc != QG_OK) return rc;
    return qg::launch_dequant_q4k(W, out, N, K, stream);
}

int qdequant_iq3(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K, cudaStream_t stream) {
    int rc = check_dequant(W, grid, true, out, N, K, 98);
    if (rc != QG_OK) return rc;
    return qg::launch_dequant_iq3(W, grid, out, N, K, stream);
}

int qdequant_iq3xxs(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K, cudaStream_t stream) {
    int rc = check_dequant(W, grid, true, out, N, K, 98);
    if (rc != QG_OK) return rc;
    return qg::launch_dequant_iq3xxs(W, grid, out, N, K, stream);
}

int qg_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return qg::cuda_fail(cudaGetLastError());
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, qg_status_word, sizeof(v)) != cudaSuccess) return qg::cuda_fail(cudaGetLastError());
    if (v != 0 && cudaMemcpyToSymbol(qg_status_word, &zero, sizeof(zero)) != cudaSuccess) return qg::cuda_fail(cudaGetLastError());
    if (v & qg::kStatusTimeout) return QG_ETIMEOUT;
    if (v & qg::kStatusBounds) return QG_EBOUNDS;
    return QG_OK;
}

int qg_test_bounded_wait(cudaStream_t stream) {
    unsigned* st = status_ptr();
    if (!st) return qg::cuda_fail(cudaGetLastError());
    qg_bounded_wait_probe<<<1, 32, 0, stream>>>(st);
    return qg::launch_status();
}

int qg_test_chain_step(const float* X, float* Y, int64_t K, int grid, unsigned flags, cudaStream_t stream) {
    if (!X || !Y || K <= 0 || K % 256 != 0 || K > (int64_t(1) << 31) || grid < 1 || grid > 65535) return QG_EINVAL;
    if (flags & ~static_cast<unsigned>(QG_PREFETCH_WEIGHTS)) return QG_EINVAL;
    if (!aligned16(X) || !aligned16(Y)) return QG_EALIGN;
    if (overlap(Y, int64_t(grid) * 32 * 4, X, K * 4)) return QG_EALIAS;
    return qg::launch_chain_step(X, Y, K, grid, flags, stream);
}

int qg_last_cuda_error(void) { return qg::t_last_cuda_error; }

const char* qg_strerror(int status) {
    switch (status) {
        case QG_OK: return "ok";
        case QG_EINVAL: return "invalid argument (M, N, K or a null pointer)";
        case QG_EALIGN: return "pointer not 16-byte aligned";
        case QG_ECUDA: return "CUDA runtime or launch error";
        case QG_ETIMEOUT: return "a bounded wait inside a kernel gave up";
        case QG_EBOUNDS: return "an index check inside a kernel failed";
        case QG_EALIAS: return "output overlaps an input";
        case QG_ESCRATCH: return "more stages than the fixed scratch of qgemv_q4k_pass_noalloc holds";
        default: return "unknown status";
    }
}

}  // extern "C"
