/*
 * CPU oracle for the block-quantised GEMV: TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the bench's CPU-baseline leg load this
 * library.  It shares no code, header or table with the CUDA library.
 *
 * Plain C99, built with -O2 -ffp-contract=off so that every float operation
 * below is rounded exactly as written (no fused multiply-add).
 *
 * Sources (page title, section):
 *   - Q4_K: page 1 "Rewriting picoLM in Python", function dequantize_q4_K
 *     (block layout, the 6-bit scale/min unpack, the nibble-to-weight map).
 *   - IQ3:  page 4 "iq3_pack.py" (colibri fmt=5), module docstring (layout,
 *     value formula) and function decode (sign words, implied 8th sign,
 *     sub-scale), function grid (the x0.5 applied to the published table).
 *   - IQ3_XXS: page 3 (llama.cpp's codebook formats as trainable students),
 *     the format table (98 bytes, d at bytes 0-1, s the top 4 bits of the
 *     uint32s at bytes 66-97, eff = d*(0.5+s)*0.5), the class Format /
 *     eff_np (eff times v, v = codebook entry times sign) and the note that
 *     IQ3_XXS stores 8 signs in 7 bits with an even count of negatives.
 *   - IQ4_NL, IQ4_XS, IQ3_S, IQ2_XXS: page 3, the format table (block and
 *     sub-block sizes, eff, byte counts, where d and s sit), get_s (how s is
 *     read), eff_np (eff = d, d*(s-32), d*(1+2s), d*(0.5+s)*0.25) and
 *     encode (the code bytes of IQ4_NL, IQ3_S and IQ2_XXS).
 *   - GEMV: page 1, model_forward / forward: matmul(out, x, W, n_in, n_out)
 *     computes out = W x with one output per row of W.
 *
 * Pins: tests/test_oracle_pins.py checks every function here against
 * hand-worked blocks (tests/golden/), exact closed forms, numpy's fp16
 * conversion and math.fsum.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 256
#define Q4K_BYTES 144
#define IQ3_BYTES 98

/* IEEE-754 binary16 -> binary32, exact, from the format's definition:
 * sign 1 bit, exponent 5 bits (bias 15), fraction 10 bits; exponent 0 is
 * zero/subnormal (value = fraction * 2^-24), exponent 31 is Inf/NaN. */
float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t expo = (uint32_t)(h >> 10) & 31u;
    uint32_t frac = (uint32_t)h & 1023u;
    float v;
    if (expo == 0) {
        v = ldexpf((float)frac, -24);           /* exact: frac < 2^10 */
    } else if (expo == 31) {
        if (frac == 0) {
            v = INFINITY;
        } else {                                /* keep the payload bits */
            uint32_t bits = 0x7f800000u | (frac << 13);
            memcpy(&v, &bits, 4);
        }
    } else {
        v = ldexpf((float)(1024u + frac), (int)expo - 25);
    }
    return sign ? -v : v;
}

void oracle_f16_to_f32_array(const uint16_t *h, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f16_to_f32(h[i]);
}

static uint16_t le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t le32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* Page 1, dequantize_q4_K: the 12 packed bytes hold eight 6-bit scales and
 * eight 6-bit mins.  j < 4: the low six bits of bytes j and j+4.  j >= 4: the
 * low (scale) or high (min) nibble of byte j+4, with the top two bits of byte
 * j-4 (scale) or byte j (min) above it. */
void oracle_q4k_scale_min(const uint8_t p[12], uint8_t sc[8], uint8_t mn[8])
{
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = (uint8_t)(p[j] & 63);
            mn[j] = (uint8_t)(p[j + 4] & 63);
        } else {
            sc[j] = (uint8_t)((p[j + 4] & 0xF) | ((p[j - 4] >> 6) << 4));
            mn[j] = (uint8_t)((p[j + 4] >> 4) | ((p[j] >> 6) << 4));
        }
    }
}

/* One Q4_K block (144 bytes) -> 256 fp32 weights, page 1 dequantize_q4_K.
 * Byte 0-1 d, 2-3 dmin (fp16), 4-15 packed scales/mins, 16-143 qs.  qs is
 * four groups of 32 bytes; in group g, byte l gives weight 64g+l from its low
 * nibble (scale/min index 2g) and weight 64g+32+l from its high nibble
 * (index 2g+1).  Each weight is (d*sc)*q - (dmin*mn), evaluated left to
 * right in fp32 as the page's numpy expression does. */
void oracle_dequant_q4k_block(const uint8_t *blk, float *out)
{
    float d = oracle_f16_to_f32(le16(blk + 0));
    float dmin = oracle_f16_to_f32(le16(blk + 2));
    uint8_t sc[8], mn[8];
    oracle_q4k_scale_min(blk + 4, sc, mn);
    const uint8_t *qs = blk + 16;
    for (int g = 0; g < 4; ++g) {
        for (int l = 0; l < 32; ++l) {
            uint8_t q = qs[32 * g + l];
            float lo = (float)(q & 0xF), hi = (float)(q >> 4);
            float a0 = d * (float)sc[2 * g];
            float a1 = a0 * lo;
            float b0 = dmin * (float)mn[2 * g];
            out[64 * g + l] = a1 - b0;
            float c0 = d * (float)sc[2 * g + 1];
            float c1 = c0 * hi;
            float e0 = dmin * (float)mn[2 * g + 1];
            out[64 * g + 32 + l] = c1 - e0;
        }
    }
}

/* One IQ3 super-block (98 bytes) -> 256 fp32 weights, page 4 decode.
 * Bytes 0-63: one grid index per 4 weights; 64-95: eight little-endian u32,
 * one per 32-weight sub-block ib: bits 7l..7l+6 are the sign bits of weights
 * 8l..8l+6 of the sub-block (bit set => negative), the sign of weight 8l+7 is
 * the XOR of those seven bits, bits 28-31 are the sub-scale code; 96-97: fp16
 * d.  value = mag * sign * db with mag = grid_byte * 0.5 (fp32, page 4 grid())
 * and db = d * (0.5 + code) * 0.5 (fp64, as numpy promotes it), rounded once
 * to fp32 when stored. */
void oracle_dequant_iq3_block(const uint8_t *blk, const uint8_t *grid, float *out)
{
    double d = (double)oracle_f16_to_f32(le16(blk + 96));
    for (int ib = 0; ib < 8; ++ib) {
        const uint8_t *idx = blk + 8 * ib;
        uint32_t word = le32(blk + 64 + 4 * ib);
        uint32_t code = (word >> 28) & 0xF;
        double db = d * (0.5 + (double)code) * 0.5;
        for (int l = 0; l < 4; ++l) {
            uint32_t seven = (word >> (7 * l)) & 0x7F;
            uint32_t par = 0;
            for (int j = 0; j < 8; ++j) {
                uint32_t neg;
                if (j < 7) {
                    neg = (seven >> j) & 1u;
                    par ^= neg;
                } else {
                    neg = par;
                }
                int t = 8 * l + j;              /* weight within the sub-block */
                uint8_t gidx = idx[t / 4];
                float mag = (float)grid[4 * gidx + (t % 4)] * 0.5f;
                float sgn = neg ? -1.0f : 1.0f;
                float ms = mag * sgn;
                out[32 * ib + t] = (float)((double)ms * db);
            }
        }
    }
}

/* One IQ3_XXS block (98 bytes) -> 256 fp32 weights, page 3.  Bytes 0-1: fp16
 * d; 2-65: one codebook index per 4 weights (the code bytes: everything but
 * d and the sub-scales); 66-97: eight little-endian u32, one per 32-weight
 * sub-block: bits 7l..7l+6 the signs of weights 8l..8l+6 (bit set =>
 * negative), the eighth sign the XOR of those seven (an even count of
 * negatives), bits 28-31 the sub-scale s.  eff = d*(0.5+s)*0.5 in fp32 (as
 * ggml computes it), v = grid entry (raw, not halved) times the sign,
 * weight = eff*v (exact in fp32: page 3 notes v*eff is exact). */
void oracle_dequant_iq3xxs_block(const uint8_t *blk, const uint8_t *grid, float *out)
{
    float d = oracle_f16_to_f32(le16(blk + 0));
    for (int ib = 0; ib < 8; ++ib) {
        const uint8_t *idx = blk + 2 + 8 * ib;
        uint32_t word = le32(blk + 66 + 4 * ib);
        float s = (float)((word >> 28) & 0xF);
        float eff = d * (0.5f + s) * 0.5f;
        for (int l = 0; l < 4; ++l) {
            uint32_t seven = (word >> (7 * l)) & 0x7F;
            uint32_t par = 0;
            for (int j = 0; j < 8; ++j) {
                uint32_t neg;
                if (j < 7) {
                    neg = (seven >> j) & 1u;
                    par ^= neg;
                } else {
                    neg = par;
                }
                int t = 8 * l + j;
                float v = (float)grid[4 * idx[t / 4] + (t % 4)];
                if (neg) v = -v;
                out[32 * ib + t] = eff * v;
            }
        }
    }
}

/* ---- page 3's other codebook formats, decoded per 256 weights ----------
 * Every one stores weight = eff * v, v = (codebook entry) * (sign), d the
 * block's fp16 scale at bytes 0-1 and s the sub-block scales; products are
 * exact in fp32 (page 3: "v*eff is exact in fp32").  The codebooks are not
 * printed on the pages; they are inputs: the IQ4 table as 16 signed bytes,
 * the IQ3_S grid as 512 x 4 bytes, the IQ2_XXS grid as 256 x 8 bytes. */

/* IQ4_NL: 32 weights in 18 bytes: d, then 16 bytes where byte i holds the
 * code of weight i in its low nibble and of weight i+16 in its high nibble
 * (page 3, encode: q[:16] | q[16:] << 4); eff = d; v = table[code].  One
 * 256-weight unit is 8 consecutive blocks (144 bytes). */
void oracle_dequant_iq4nl_unit(const uint8_t *u, const int8_t *table, float *out)
{
    for (int b = 0; b < 8; ++b) {
        const uint8_t *blk = u + 18 * b;
        float d = oracle_f16_to_f32(le16(blk));
        for (int i = 0; i < 16; ++i) {
            uint8_t q = blk[2 + i];
            out[32 * b + i] = d * (float)table[q & 0xF];
            out[32 * b + 16 + i] = d * (float)table[q >> 4];
        }
    }
}

/* IQ4_XS: 256 weights in 136 bytes: d at 0-1; s of sub-block j (6 bits) =
 * nibble j of bytes 4-7 (low nibble first: page 3 get_s's _nibbles) plus
 * bits 2j, 2j+1 of the little-endian u16 at bytes 2-3 as bits 4-5;
 * eff = d * (s - 32); v = table[code].  The code bytes are bytes 8-135,
 * 16 per 32-weight sub-block, packed as in IQ4_NL (low nibble weight i,
 * high nibble weight i+16): the pages do not print IQ4_XS's code layout,
 * this is the reading that shares IQ4_NL's codebook and packing. */
void oracle_dequant_iq4xs_unit(const uint8_t *u, const int8_t *table, float *out)
{
    float d = oracle_f16_to_f32(le16(u));
    uint16_t sh = le16(u + 2);
    for (int j = 0; j < 8; ++j) {
        int lo = (u[4 + j / 2] >> (4 * (j & 1))) & 0xF;
        int hi = (sh >> (2 * j)) & 3;
        int s = lo | (hi << 4);
        float eff = d * (float)(s - 32);
        const uint8_t *qs = u + 8 + 16 * j;
        for (int i = 0; i < 16; ++i) {
            out[32 * j + i] = eff * (float)table[qs[i] & 0xF];
            out[32 * j + 16 + i] = eff * (float)table[qs[i] >> 4];
        }
    }
}

/* IQ3_S: 256 weights in 110 bytes: d; bytes 2-65 the low 8 bits of the 64
 * grid indices (one per 4 weights); bytes 66-73 their 9th bits, index i at
 * bit i%8 of byte 66+i/8 (packbits, little bit order); bytes 74-105 one
 * sign bit per weight, weight k at bit k%8 of byte 74+k/8 (set = negative);
 * bytes 106-109 the eight 4-bit s, sub-block j in nibble j (low first);
 * eff = d * (1 + 2s); v = grid[index][k%4] * sign (page 3, encode, get_s). */
void oracle_dequant_iq3s_unit(const uint8_t *u, const uint8_t *grid, float *out)
{
    float d = oracle_f16_to_f32(le16(u));
    for (int j = 0; j < 8; ++j) {
        int s = (u[106 + j / 2] >> (4 * (j & 1))) & 0xF;
        float eff = d * (float)(1 + 2 * s);
        for (int t = 0; t < 32; ++t) {
            int k = 32 * j + t;
            int gi = k / 4;
            int idx = u[2 + gi] | (((u[66 + gi / 8] >> (gi % 8)) & 1) << 8);
            float v = (float)grid[4 * idx + (k % 4)];
            if ((u[74 + k / 8] >> (k % 8)) & 1) v = -v;
            out[k] = eff * v;
        }
    }
}

/* IQ2_XXS: 256 weights in 66 bytes: d; then per 32-weight sub-block j two
 * little-endian u32 at 2+8j: the first holds the grid indices of its four
 * 8-weight groups (byte g), the second the groups' 7-bit sign fields at bits
 * 7g..7g+6 (bit i set = weight i of the group negative; the eighth sign is
 * their parity, an even count of negatives) and s in bits 28-31;
 * eff = d * (0.5 + s) * 0.25; v = grid[index][i] * sign (page 3, encode,
 * get_s, the even-sign note). */
void oracle_dequant_iq2xxs_unit(const uint8_t *u, const uint8_t *grid, float *out)
{
    float d = oracle_f16_to_f32(le16(u));
    for (int j = 0; j < 8; ++j) {
        uint32_t aux0 = le32(u + 2 + 8 * j), aux1 = le32(u + 6 + 8 * j);
        float s = (float)((aux1 >> 28) & 0xF);
        float eff = d * (0.5f + s) * 0.25f;
        for (int g = 0; g < 4; ++g) {
            uint32_t idx = (aux0 >> (8 * g)) & 0xFF;
            uint32_t seven = (aux1 >> (7 * g)) & 0x7F, par = 0;
            for (int i = 0; i < 8; ++i) {
                uint32_t neg;
                if (i < 7) {
                    neg = (seven >> i) & 1u;
                    par ^= neg;
                } else {
                    neg = par;
                }
                float v = (float)grid[8 * idx + i];
                if (neg) v = -v;
                out[32 * j + 8 * g + i] = eff * v;
            }
        }
    }
}

/* Bytes per 256-weight unit of the formats above (fmt 3..6). */
static int64_t cb_unit_bytes(int fmt)
{
    return fmt == 3 ? 144 : fmt == 4 ? 136 : fmt == 5 ? 110 : 66;
}

static void cb_unit(int fmt, const uint8_t *u, const uint8_t *tab, float *out)
{
    if (fmt == 3) oracle_dequant_iq4nl_unit(u, (const int8_t *)tab, out);
    else if (fmt == 4) oracle_dequant_iq4xs_unit(u, (const int8_t *)tab, out);
    else if (fmt == 5) oracle_dequant_iq3s_unit(u, tab, out);
    else oracle_dequant_iq2xxs_unit(u, tab, out);
}

void oracle_dequant_cb(int fmt, const uint8_t *W, const uint8_t *tab, int64_t N, int64_t K, float *out)
{
    int64_t nb = K / QK, ub = cb_unit_bytes(fmt);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            cb_unit(fmt, W + (n * nb + b) * ub, tab, out + n * K + b * QK);
}

/* Whole rows: W is [N][K/256 blocks], out is [N][K] fp32. */
void oracle_dequant_q4k(const uint8_t *W, int64_t N, int64_t K, float *out)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            oracle_dequant_q4k_block(W + (n * nb + b) * Q4K_BYTES, out + n * K + b * QK);
}

void oracle_dequant_iq3(const uint8_t *W, const uint8_t *grid, int64_t N, int64_t K, float *out)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            oracle_dequant_iq3_block(W + (n * nb + b) * IQ3_BYTES, grid, out + n * K + b * QK);
}

void oracle_dequant_iq3xxs(const uint8_t *W, const uint8_t *grid, int64_t N, int64_t K, float *out)
{
    int64_t nb = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            oracle_dequant_iq3xxs_block(W + (n * nb + b) * IQ3_BYTES, grid, out + n * K + b * QK);
}

/* GEMV reference for selected rows.  Y[m][r] = sum_k (double)w[row][k] * (double)x[m][k],
 * summed in k order in fp64; A[m][r] = sum_k |w*x| in fp64 (the scale of the
 * tolerance).  rows == NULL means rows 0..nrows-1.  Y and A are [M][nrows].
 * fmt 0 = Q4_K, 1 = IQ3 (page 4), 2 = IQ3_XXS, 3 = IQ4_NL, 4 = IQ4_XS,
 * 5 = IQ3_S, 6 = IQ2_XXS (page 3; grid = the format's codebook).  Rows are independent; with nthreads > 1 they are
 * split across OpenMP threads (each row's sum is still sequential). */
static void gemv_rows(int fmt, const uint8_t *W, const uint8_t *grid, const float *X,
                      int M, int64_t K, const int64_t *rows, int64_t nrows,
                      double *Y, double *A, int nthreads)
{
    int64_t nb = K / QK;
    int64_t bytes = fmt == 0 ? Q4K_BYTES : fmt <= 2 ? IQ3_BYTES : cb_unit_bytes(fmt);
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        float w[QK];
        int64_t row = rows ? rows[r] : r;
        for (int m = 0; m < M; ++m) {
            Y[(int64_t)m * nrows + r] = 0.0;
            A[(int64_t)m * nrows + r] = 0.0;
        }
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = W + (row * nb + b) * bytes;
            if (fmt == 0)
                oracle_dequant_q4k_block(blk, w);
            else if (fmt == 1)
                oracle_dequant_iq3_block(blk, grid, w);
            else if (fmt == 2)
                oracle_dequant_iq3xxs_block(blk, grid, w);
            else
                cb_unit(fmt, blk, grid, w);
            for (int m = 0; m < M; ++m) {
                const float *x = X + (int64_t)m * K + b * QK;
                double y = Y[(int64_t)m * nrows + r], a = A[(int64_t)m * nrows + r];
                for (int k = 0; k < QK; ++k) {
                    double p = (double)w[k] * (double)x[k];
                    y += p;
                    a += fabs(p);
                }
                Y[(int64_t)m * nrows + r] = y;
                A[(int64_t)m * nrows + r] = a;
            }
        }
    }
}

void oracle_gemv_q4k(const uint8_t *W, const float *X, int M, int64_t K,
                     const int64_t *rows, int64_t nrows, double *Y, double *A, int nthreads)
{
    gemv_rows(0, W, NULL, X, M, K, rows, nrows, Y, A, nthreads);
}

void oracle_gemv_iq3(const uint8_t *W, const uint8_t *grid, const float *X, int M, int64_t K,
                     const int64_t *rows, int64_t nrows, double *Y, double *A, int nthreads)
{
    gemv_rows(1, W, grid, X, M, K, rows, nrows, Y, A, nthreads);
}

void oracle_gemv_iq3xxs(const uint8_t *W, const uint8_t *grid, const float *X, int M, int64_t K,
                        const int64_t *rows, int64_t nrows, double *Y, double *A, int nthreads)
{
    gemv_rows(2, W, grid, X, M, K, rows, nrows, Y, A, nthreads);
}

void oracle_gemv_cb(int fmt, const uint8_t *W, const uint8_t *tab, const float *X, int M, int64_t K,
                    const int64_t *rows, int64_t nrows, double *Y, double *A, int nthreads)
{
    gemv_rows(fmt, W, tab, X, M, K, rows, nrows, Y, A, nthreads);
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
