/*
 * qgemv: fused-dequantisation GEMV over block-quantised weights (sm_103a).
 *
 * C ABI of libqgemv.so.  Plain pointers and sizes only.
 *
 * The operation (page 1 "Rewriting picoLM in Python", model_forward /
 * forward: matmul(out, x, W, n_in, n_out, type) with one output per weight
 * row) is
 *
 *     Y[m][n] = sum_k w[n][k] * X[m][k]      0 <= m < M, 0 <= n < N, 0 <= k < K
 *
 * where w is decoded on the fly from the quantised bytes and never stored.
 *
 * Layouts (all little-endian, no padding):
 *   W  row n, then super-block b (256 weights each): byte offset (n*K/256 + b)*B
 *      with B = 144 for Q4_K, 98 for IQ3.
 *   X  [M][K] fp32, row-major.     Y  [M][N] fp32, row-major (written, not
 *      accumulated): Y = X * W^T, the layout of torch.nn.functional.linear.
 *
 * Block formats:
 *   Q4_K (page 1, dequantize_q4_K): fp16 d @0, fp16 dmin @2, 12 bytes of
 *     packed 6-bit scales/mins @4 (fields j >= 4 straddle bytes), 128 nibble
 *     bytes @16; weight = d*sc*q - dmin*mn.
 *   IQ3 (page 4 "iq3_pack.py", fmt=5, module docstring and decode): 64 grid
 *     index bytes @0, eight u32 @64 (per 32-weight sub-block: four 7-bit sign
 *     words in bits 0-27, the 8th sign of each 8-group the XOR of its seven
 *     stored signs, a 4-bit code in bits 28-31), fp16 d @96;
 *     weight = d*(0.5+code)*0.5 * grid[idx][j]*0.5 * sign.
 *
 * Ownership: every pointer is caller-owned device memory; the library
 * allocates nothing per call.  Calls are asynchronous on `stream` (0 = the
 * legacy default stream).  Y must not overlap W, X or grid.
 *
 * Errors: functions return QG_OK (0) or a negative QG_E* code and never
 * abort, throw or trap.  Argument errors are detected on the host before any
 * launch.  Faults detected inside a kernel (a bounded wait that gave up) are
 * latched in a per-device status word; qg_device_status reports and clears
 * it.  After QG_ECUDA, qg_last_cuda_error gives the CUDA error behind it.
 *
 * Threads: every entry point may be called from several host threads at
 * once (each on its own stream, or ordered by the caller); the library's
 * per-device set-up is done once and shared.  The device is the calling
 * thread's current CUDA device.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QG_OK 0
#define QG_EINVAL (-1)    /* K % 256 != 0, M outside [1, 32], N <= 0, K <= 0, null pointer */
#define QG_EALIGN (-2)    /* W, X, Y or grid not 16-byte aligned */
#define QG_ECUDA (-3)     /* a CUDA runtime call or kernel launch failed */
#define QG_ETIMEOUT (-4)  /* device: a bounded wait inside a kernel gave up */
#define QG_EBOUNDS (-5)   /* device: an index check inside a kernel failed */
#define QG_EALIAS (-6)    /* Y overlaps W, X or grid */
#define QG_ESCRATCH (-7)  /* request larger than the fixed scratch of qgemv_q4k_pass_noalloc */

#define QG_MAX_M 32
#define QG_MAX_GROUP 4

/* Launch flag for the *_ex entry points.  QG_PREFETCH_WEIGHTS promises that W
 * (and the IQ3 grid, and a fused call's RMSNorm weight) are not written by
 * the kernel that precedes this call in the stream.  The GEMV is then launched as a programmatic dependent launch:
 * it may start while the preceding kernel is still running and stream its
 * first weight tiles, and it waits for the preceding kernel to complete (all
 * its memory visible) before it reads X or writes Y.  Without the flag the
 * call is ordinary stream-ordered work. */
#define QG_PREFETCH_WEIGHTS 1u

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

/* Q4_K GEMV, 1 <= M <= 32.
 * Page 1 "Rewriting picoLM in Python", dequantize_q4_K (format) and
 * model_forward's matmul (operation).
 * W: N*K/256*144 bytes.  X: M*K floats.  Y: M*N floats (output).
 * Numerics: |Y - exact| <= 1e-5 * sum_k |w*x| per element.
 * Each 32-weight sub-block is summed as a*sum((q - c)*x) - (b - a*c)*sum(x),
 * a = d*sc, b = dmin*mn, c the integer in [0, 15] nearest b/a, so sub-blocks
 * whose d*sc*q and dmin*mn cancel keep that accuracy (a row of zero weights
 * gives exactly 0).  Up to 4 tokens: the fp32 FMA path; range: every finite
 * x (slices of 256 x values whose largest |x| lies outside [2^-24, 2^39)
 * take a slower rescaled decode, a power of two in, its inverse out), so the
 * outputs are only limited by fp32 itself.  From 5 tokens: the tcgen05
 * tensor cores in groups of 5 to 10 tokens, each streaming W once, with the
 * same factoring: q - c enters the MMA exactly (bf16) and x split exactly
 * into three bf16 parts, so every product is exact and the sums are fp32 in
 * tensor memory; there x is multiplied as given (|x| within [2^-100,
 * 2^100]), Y is zeroed on `stream` and row sums that different CTAs share
 * are added with fp32 atomics, so repeated calls may differ in the last
 * bits.  The same holds for qgemv_q4k_group; qgemv_q4k_fused (its RMSNorm
 * prologue sums x^2 in fp32: |x| below 2^63) and qgemv_q4k_pass keep the
 * FMA path. */
QG_API int qgemv_q4k(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t stream);

/* qgemv_q4k with launch flags (0 or QG_PREFETCH_WEIGHTS); other flag bits:
 * QG_EINVAL. */
QG_API int qgemv_q4k_ex(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, unsigned flags,
                        cudaStream_t stream);

/* IQ3 (98-byte super-block) GEMV, 1 <= M <= 32, within 1e-5 * sum|w*x|.
 * Page 4 "iq3_pack.py", module docstring and decode (format); page 1
 * model_forward's matmul (operation).
 * grid: 256*4 bytes, the codebook in the published doubled units (the kernel
 * applies the 0.5 of page 4's grid()).  Other arguments as qgemv_q4k.
 * K/256 a multiple of 8: M <= 4 takes the fp32 FMA tensor-map path; M >= 5
 * the tcgen05 tensor cores in groups of 5 to 10 tokens, each streaming W
 * once: the signed grid bytes enter the MMA exactly (bf16), x split exactly
 * into three bf16 parts, so every product is exact and the sums are fp32 in
 * tensor memory, each sub-block factor applied afterwards.  There Y is
 * zeroed on `stream` and row sums that different CTAs share are added with
 * fp32 atomics, so repeated calls may differ in the last bits.  Other K
 * take a slower byte-addressed fp32 path (groups of 8 tokens).  Range: the
 * FMA tensor-map path takes every finite x (columns whose largest |x| lies
 * outside [2^-24, 2^39) are rescaled by a power of two); the tensor-core and
 * byte-addressed paths multiply x as given, so there |x| must stay within
 * [2^-100, 2^100] for the tolerance to hold. */
QG_API int qgemv_iq3(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
              cudaStream_t stream);

/* qgemv_iq3 with launch flags (0 or QG_PREFETCH_WEIGHTS). */
QG_API int qgemv_iq3_ex(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                        unsigned flags, cudaStream_t stream);

/* IQ3_XXS GEMV: the same 98-byte super-block in page 3's byte order and
 * scale convention (llama.cpp's IQ3_XXS; page 3, the format table, Format
 * and eff_np): fp16 d @0, 64 grid index bytes @2, eight u32 @66 (sign
 * fields and implied eighth sign as qgemv_iq3, the 4-bit sub-scale s in
 * bits 28-31); weight = d*(0.5+s)*0.5 * grid[idx][j] * sign, the grid
 * entries used as they are (no halving).  The same fields in page 4's order
 * give half these values.  Other arguments, paths and numerics as qgemv_iq3. */
QG_API int qgemv_iq3xxs(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N, int64_t K,
                        cudaStream_t stream);

/* qgemv_iq3xxs with launch flags (0 or QG_PREFETCH_WEIGHTS). */
QG_API int qgemv_iq3xxs_ex(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N,
                           int64_t K, unsigned flags, cudaStream_t stream);

/* Page 3's other codebook formats (llama.cpp's codebook formats as
 * trainable students: the format table, get_s, eff_np, encode).  Every one
 * stores weight = eff * v with v = codebook entry * sign, d the block's
 * fp16 scale at bytes 0-1; bytes per 256 weights and codebook (an input,
 * since the pages do not print it):
 *   QG_CB_IQ4_NL   144 (eight 18-byte blocks of 32 weights: d, then byte i =
 *                  code of weight i | code of weight i+16 << 4); eff = d;
 *                  codebook: 16 int8 values
 *   QG_CB_IQ4_XS   136: d; u16 @2 = bits 4-5 of the eight 6-bit s (2 per
 *                  sub-block); @4-7 their low nibbles (sub-block j: nibble j,
 *                  low first); @8-135 the codes, 16 bytes per 32-weight
 *                  sub-block packed as IQ4_NL; eff = d*(s-32); codebook as
 *                  IQ4_NL (the code layout is not printed on the pages; this
 *                  is the reading that shares IQ4_NL's packing)
 *   QG_CB_IQ3_S    110: d; @2-65 low 8 bits of the 64 grid indices (one per
 *                  4 weights); @66-73 their 9th bits (index i: bit i%8 of byte
 *                  66+i/8); @74-105 one sign bit per weight (weight k: bit k%8
 *                  of byte 74+k/8, set = negative); @106-109 the 4-bit s
 *                  (sub-block j: nibble j, low first); eff = d*(1+2s);
 *                  codebook: 512 x 4 bytes
 *   QG_CB_IQ2_XXS  66: d; per 32-weight sub-block j two u32 at 2+8j: the grid
 *                  indices of its four 8-weight groups (byte g), then the
 *                  groups' 7-bit sign fields (bits 7g..7g+6, the eighth sign
 *                  their parity: an even count of negatives) and s in bits
 *                  28-31; eff = d*(0.5+s)*0.25; codebook: 256 x 8 bytes
 * W [N][K/256 units], X [M][K], Y [M][N] as qgemv_q4k; 1 <= M <= 32;
 * codebook device memory, 16-byte aligned.  fp32 FMA path, tolerance
 * 1e-5 * sum|w*x|.  Rows that are a multiple of 16 bytes (IQ4_NL always,
 * IQ4_XS for even K/256, IQ3_S and IQ2_XXS for K/256 a multiple of 8)
 * stream through tensor-map copies; the others are read directly.  Range
 * of x: IQ3_S and IQ2_XXS on the tensor-map path take every finite x
 * (columns whose largest |x| lies outside [2^-24, 2^39) are rescaled by a
 * power of two); otherwise x is multiplied as given and |x| must stay
 * within [2^-100, 2^100].  Errors as qgemv_q4k, plus QG_EINVAL for an
 * unknown format. */
#define QG_CB_IQ4_NL 1
#define QG_CB_IQ4_XS 2
#define QG_CB_IQ3_S 3
#define QG_CB_IQ2_XXS 4
QG_API int qgemv_codebook(int format, const uint8_t* W, const void* codebook, const float* X, float* Y, int M,
                          int64_t N, int64_t K, cudaStream_t stream);

/* Test-only: dequantise a codebook-format matrix to fp32 out[N][K] (exact). */
QG_API int qdequant_codebook(int format, const uint8_t* W, const void* codebook, float* out, int64_t N, int64_t K,
                             cudaStream_t stream);

/* Several Q4_K GEMVs that read the same X (in a decode step: q, k and v of a
 * layer read the attention-norm output; gate and up read the FFN-norm
 * output) in one launch: Y[i] = X * dequant(W[i])^T for i < count,
 * 1 <= count <= QG_MAX_GROUP.  W, Y and N are HOST arrays holding device
 * pointers and row counts; Y[i] is [M][N[i]].  Same K for every matrix.
 * Results are identical to count separate qgemv_q4k_ex calls (from 5
 * tokens, the tensor-core path, each matrix is its own launch and the two
 * agree up to the order of the fp32 atomics).  Page 1
 * "Rewriting picoLM in Python", model_forward (the q/k/v and gate/up
 * matmuls of one layer consume the same normalised activation). */
QG_API int qgemv_q4k_group(const uint8_t* const* W, float* const* Y, const int64_t* N, int count, const float* X,
                           int M, int64_t K, unsigned flags, cudaStream_t stream);

/* IQ3 counterpart of qgemv_q4k_group; one grid for all matrices.  From 5
 * tokens (the tensor-core path of qgemv_iq3) each matrix is its own launch
 * and results match separate calls up to the order of the fp32 atomics. */
QG_API int qgemv_iq3_group(const uint8_t* const* W, float* const* Y, const int64_t* N, int count,
                           const uint8_t* grid, const float* X, int M, int64_t K, unsigned flags,
                           cudaStream_t stream);

/* Fused prologue and epilogue of a Q4_K GEMV inside a decode step.
 * Page 2 "Candle", RmsNorm::forward (x * (1/sqrt(mean(x^2) + eps)) * weight)
 * and Block::forward (h = norm(x); x + attn(h); down(silu(gate(h)) * up(h));
 * the residual adds); page 1 model_forward (rmsnorm before the q/k/v
 * matmuls and before the output projection).  With h the GEMV input:
 *   no prologue:   h = X
 *   norm_weight:   h[m][k] = X[m][k] / sqrt(mean_k' X[m][k']^2 + norm_eps) * norm_weight[k]
 *   up:            h[m][k] = silu(X[m][k]) * up[m][k],  silu(z) = z / (1 + exp(-z))
 *   Y[i][m][n] = sum_k dequant(W[i])[n][k] * h[m][k]   (+ residual[i][m][n])
 * All pointers device, 16-byte aligned, caller-owned; NULL disables an
 * operand.  norm_weight [K] fp32; up [M][K] fp32; residual[i] [M][N[i]]
 * fp32, which may be exactly Y[i] (in-place add) but must not otherwise
 * overlap any Y.  At most one of norm_weight and up; with either, M <= 4.
 * Numerics: |Y - exact| <= 1e-5 * sum_k |w*h| per element (h exact), plus
 * the fp32 rounding of the residual add; 1/sqrt, exp and the SiLU division
 * use the fast hardware paths (a few ulp each). */
typedef struct qg_fuse {
    const float* norm_weight;
    float norm_eps;                      /* >= 0, finite */
    const float* up;
    const float* residual[QG_MAX_GROUP]; /* per matrix of a group; [0] for single calls */
} qg_fuse;

/* Q4_K GEMV with the prologue / epilogue of `fuse` (NULL: plain GEMV).
 * Same arguments, layouts and flags as qgemv_q4k_ex; fuse->residual[i] for
 * i >= 1 must be NULL.  Errors: QG_EINVAL for both prologues, a prologue
 * with M > 4, a negative or non-finite norm_eps; QG_EALIGN; QG_EALIAS. */
QG_API int qgemv_q4k_fused(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K,
                           const qg_fuse* fuse, unsigned flags, cudaStream_t stream);

/* qgemv_q4k_group with the prologue / epilogue of `fuse` (the prologue is
 * shared by the matrices, residual[i] belongs to matrix i).  In a decode
 * step: q/k/v with the attention RMSNorm, gate/up with the FFN RMSNorm. */
QG_API int qgemv_q4k_fused_group(const uint8_t* const* W, float* const* Y, const int64_t* N, int count,
                                 const float* X, int M, int64_t K, const qg_fuse* fuse, unsigned flags,
                                 cudaStream_t stream);

/* One stage of a decode pass: a group of matrices reading the same X. */
#define QG_MAX_PASS_STAGES 96
typedef struct qg_stage {
    const uint8_t* W[QG_MAX_GROUP]; /* device, Q4_K, [N[i]][K/256 blocks] */
    float* Y[QG_MAX_GROUP];         /* device, [M][N[i]] */
    int64_t N[QG_MAX_GROUP];
    int count;                      /* 1..QG_MAX_GROUP */
    const float* X;                 /* device, [M][K]; may be a Y of an earlier stage */
    int64_t K;
} qg_stage;

/* A sequence of dependent Q4_K GEMV stages (a decode pass: per layer q/k/v,
 * o, gate/up, down, then the output projection) in one persistent,
 * cooperative launch.  Stage s reads its X only after every stage < s has
 * written all of its Y, so X of a stage may be any Y of an earlier stage;
 * the weights of later stages stream while earlier stages finish.
 * Each stage meets the same tolerance as qgemv_q4k_group.  Results are
 * identical to it bit for bit where the grouped launch also decodes a
 * tile's K chunks in one CTA (one 32-row tile per CTA and one K chunk, or
 * more tiles than the SMs can each take one of); where it splits a tile's K
 * chunks over a cluster (few tiles, 2 to 8 chunks) the partial sums meet in
 * another order.  1 <= M <= 4,
 * 1 <= nstages <= QG_MAX_PASS_STAGES.  `stages` is a host array.
 * sync: caller-owned device memory of at least 4*nstages bytes (4-byte
 * aligned) used for the stage completion counts; the call zeroes it on the
 * stream; concurrent calls must not share it.  Page 1 "Rewriting picoLM in
 * Python", model_forward (the per-layer matmul sequence). */
QG_API int qgemv_q4k_pass(const qg_stage* stages, int nstages, int M, unsigned* sync, cudaStream_t stream);

/* qgemv_q4k_pass without any allocation: for callers that cannot call
 * cudaMalloc.  Examples are a plugin that its host application hands only
 * input and output buffers while the application's own pool owns the rest
 * of device memory, and a decode loop that must not stall, since cudaMalloc
 * and cudaFree may synchronise the device.  Such callers still pass all
 * inputs and outputs; only the stage completion counts (the `sync` words of
 * qgemv_q4k_pass) move into a fixed scratch array inside this library,
 * QG_NOALLOC_SCRATCH_WORDS 32-bit words (384 bytes) that every GPU which
 * loads the library holds until the process exits.  Everything else is as
 * in qgemv_q4k_pass: same stages, same results, 1 <= M <= 4.
 * nstages > QG_NOALLOC_SCRATCH_WORDS returns QG_ESCRATCH; nstages < 1,
 * M outside [1, 4] or a null `stages` returns QG_EINVAL.
 * The first call on a device, with that device current, looks up the
 * scratch array's device address; make that first call before any stream
 * capture.  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.  Each call zeroes the counts it uses on the
 * stream before its launch (the array keeps the previous call's contents).
 * All calls on a device share the one array, so calls that overlap on the
 * GPU (other streams, other host threads) race: one call can zero the
 * counts another is still using, so they give wrong results and may also
 * end in QG_ETIMEOUT (reported by qg_device_status) after a count wait gives
 * up; once one has, the call's remaining count waits return at once, so the
 * call still ends within about one wait limit (2 s).  Order such calls on
 * one stream or synchronise between them.
 * The scratch address is cached per device for the life of the process: do
 * not call the library again on a device after cudaDeviceReset (the same
 * holds for every entry point, which caches the status word's address).
 * The pages have no counterpart: this entry point exists only for callers
 * that cannot allocate. */
#define QG_NOALLOC_SCRATCH_WORDS 96
QG_API int qgemv_q4k_pass_noalloc(const qg_stage* stages, int nstages, int M, cudaStream_t stream);

/* Batched Q4_K GEMM for decode batches, 1 <= M <= 32.
 * Same operation and layouts as qgemv_q4k.  M < 16 runs the paths of
 * qgemv_q4k (tolerance 1e-5 * sum|w*x|); M >= 16 dequantises W tiles to bf16 (round to
 * nearest even) in shared memory and multiplies on the tcgen05 tensor cores
 * with fp32 accumulation in tensor memory, X also rounded to bf16
 * (tolerance 4e-3 * sum|w*x|, for |x| within [2^-100, 2^100]: bf16 keeps
 * fp32's exponent range but not its subnormals).  On this path Y is zeroed on `stream` and the
 * row sums of K ranges that different CTAs share are added into it with fp32
 * atomics, so repeated calls may differ in the last bits (the FMA path is
 * deterministic). */
QG_API int qgemm_q4k_batched(const uint8_t* W, const float* X, float* Y, int M, int64_t N, int64_t K, cudaStream_t stream);

/* Batched IQ3 GEMM for decode batches, 1 <= M <= 32.  Same operation,
 * layouts and grid as qgemv_iq3.  M >= 16 with K/256 a multiple of 8 runs
 * on the tcgen05 tensor cores with the weights exact: the signed grid bytes
 * in bf16, each sub-block factor d*(0.5+code)*0.25 (page 4 "iq3_pack.py",
 * decode) applied in fp32 to the sub-block's sums afterwards, X rounded to
 * bf16 (tolerance 4e-3 * sum|w*x|; fp32 atomics as in qgemm_q4k_batched, so
 * not bit-reproducible); otherwise the paths of qgemv_iq3 (1e-5 *
 * sum|w*x|). */
QG_API int qgemm_iq3_batched(const uint8_t* W, const uint8_t* grid, const float* X, float* Y, int M, int64_t N,
                             int64_t K, cudaStream_t stream);

/* Test-only: dequantise a Q4_K matrix to fp32 out[N][K] (caller-owned device
 * memory, N*K floats), bit-exact with page 1's fp32 evaluation order
 * ((d*sc)*q - (dmin*mn), each operation rounded). */
QG_API int qdequant_q4k(const uint8_t* W, float* out, int64_t N, int64_t K, cudaStream_t stream);

/* Test-only: dequantise an IQ3 matrix to fp32 out[N][K]; every value is
 * exact (at most 24 significant bits), hence bit-exact with page 4's decode. */
QG_API int qdequant_iq3(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K, cudaStream_t stream);

/* Test-only: dequantise an IQ3_XXS matrix (page 3 order) to fp32 out[N][K];
 * exact like qdequant_iq3. */
QG_API int qdequant_iq3xxs(const uint8_t* W, const uint8_t* grid, float* out, int64_t N, int64_t K,
                           cudaStream_t stream);

/* Synchronise `stream`, then return and clear the current device's status
 * word: QG_OK, QG_ETIMEOUT or QG_EBOUNDS (QG_ECUDA if the sync failed). */
QG_API int qg_device_status(cudaStream_t stream);

/* Test-only fault check: launches a kernel whose mbarrier wait can never
 * complete (nothing arrives on it); the wait gives up after a bounded number
 * of polls, records QG_ETIMEOUT in the status word and the kernel returns.
 * Never traps or hangs. */
QG_API int qg_test_bounded_wait(cudaStream_t stream);

/* Test-only measurement aid: one launch that does only what a GEMV of a
 * decode step must do on the dependency chain: with QG_PREFETCH_WEIGHTS it
 * is a programmatic dependent launch that lets the next launch start and
 * waits for the previous one; then each of `grid` CTAs reads X[0..K) (fp32)
 * and writes 32 floats of Y (Y holds grid*32 floats; caller-owned device
 * memory, 16-byte aligned, not overlapping X).  A chain of these with the
 * grids of a step's GEMVs measures the step's dependent-launch floor.  The
 * pages have no counterpart. */
QG_API int qg_test_chain_step(const float* X, float* Y, int64_t K, int grid, unsigned flags, cudaStream_t stream);

/* Static description of a status code. */
QG_API const char* qg_strerror(int status);

/* The cudaError_t of the CUDA runtime call behind the calling host thread's
 * most recent QG_ECUDA (0 if that failure was not a runtime call, e.g. a
 * tensor-map encoding; 0 before any).  Per host thread; other status codes
 * leave it unchanged. */
QG_API int qg_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
