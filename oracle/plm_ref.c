/*
 * ORACLE -- test infrastructure only.  Plain, slow, scalar C99 statement of
 * what the packed-weight matmul `gemm_quant` computes.  Only the tests, the
 * smoke check and the bench's CPU-baseline leg may call it; the product path
 * never does.  It shares no code with the CUDA library.
 *
 * Sources (PocketLLM pages):
 *  - "What it runs" section of the PocketLLM README: K-quant weights are
 *    decoded inside the matmul, never widened; q4_K is served by packed int8
 *    activation kernels built on the format's own group arithmetic.
 *  - "Current status" table, row "src/ -- the C++ engine" (the Korean rewrite
 *    of the README): the CPU gemm_quant quantizes the activations to int8 the
 *    llama.cpp way, one 256-element block per task; q4_K sub-blocks may be
 *    summed in int16, q6_K sub-blocks may not (the output head stays on the
 *    int32 row path).
 *  - The block layouts are the public GGML K-quant formats the pages name:
 *      q4_K (144 B / 256 w): f16 d, f16 dmin, u8 scales[12] holding eight
 *           6-bit (scale, min) pairs, u8 qs[128]; each 64-weight chunk keeps
 *           its first 32 weights in the low nibbles and the next 32 in the
 *           high nibbles; weight = d*sc_j*q - dmin*m_j.
 *      q5_K (176 B / 256 w): as q4_K plus a fifth bit per weight: f16 d,
 *           f16 dmin, u8 scales[12], u8 qh[32], u8 qs[128]; weight 64c + l
 *           (l < 32) takes qs[32c + l] & 15 and bit 2c of qh[l], weight
 *           64c + 32 + l takes qs[32c + l] >> 4 and bit 2c + 1 of qh[l];
 *           q5 = nibble + 16 * bit, weight = d*sc_j*q5 - dmin*m_j.
 *      q6_K (210 B / 256 w): u8 ql[128], u8 qh[64], i8 scales[16] (one per
 *           16 weights), f16 d; weight = d*sc*(q6 - 32).
 *      q8_K (292 B / 256 x): f32 d, i8 qs[256], i16 bsums[16].
 *    q8_K quantization: signed amax, iscale = -128/max, nearest integer,
 *    clamp to 127, d = 1/iscale, one bsum per 16 values.
 *
 * Readings taken where the pages are silent (all stated again in the design
 * notes): nearest integer is round-half-to-even; the amax tie goes to the
 * first occurrence and keeps its sign; an all-zero chunk gives d = 0 and
 * zero codes; Y is overwritten, Y[i][r] = sum over k of x_i . w_r.
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off (no fast-math), optional OpenMP
 * over output rows only.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 256
#define Q4K_BYTES 144
#define Q5K_BYTES 176
#define Q6K_BYTES 210
#define Q8K_BYTES 292

/* ------------------------------------------------------------------ */
/* IEEE 754 binary16 -> binary32, exact, from the bit fields.          */
/* ------------------------------------------------------------------ */
float plm_ref_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t expo = (uint32_t)(h >> 10) & 31u;
    uint32_t mant = (uint32_t)h & 1023u;
    float mag;
    if (expo == 0) {
        mag = ldexpf((float)mant, -24);                 /* zero / subnormal */
    } else if (expo == 31) {
        mag = mant == 0 ? INFINITY : NAN;
    } else {
        mag = ldexpf((float)(1024u + mant), (int)expo - 25);
    }
    return sign ? -mag : mag;
}

static float load_f16(const uint8_t* p) {
    return plm_ref_f16_to_f32((uint16_t)(p[0] | ((uint16_t)p[1] << 8)));
}
static float load_f32(const uint8_t* p) { float v; memcpy(&v, p, 4); return v; }
static int16_t load_i16(const uint8_t* p) { int16_t v; memcpy(&v, p, 2); return v; }

/* ------------------------------------------------------------------ */
/* q8_K activation quantization, one 256-element chunk at a time.      */
/* ------------------------------------------------------------------ */
static int round_half_even(float v) {
    float r = nearbyintf(v);         /* default FP environment: to nearest, ties to even */
    return (int)r;
}

static void quantize_chunk(const float* x, uint8_t* blk) {
    float amax = 0.0f, max = 0.0f;
    for (int i = 0; i < QK; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) { amax = a; max = x[i]; }
    }
    float d;
    int8_t qs[QK];
    int16_t bsums[16];
    if (amax == 0.0f) {
        d = 0.0f;
        memset(qs, 0, sizeof qs);
        memset(bsums, 0, sizeof bsums);
    } else {
        float iscale = -128.0f / max;
        for (int i = 0; i < QK; ++i) {
            float t = iscale * x[i];
            int q = round_half_even(t);
            if (q > 127) q = 127;
            qs[i] = (int8_t)q;
        }
        for (int g = 0; g < 16; ++g) {
            int s = 0;
            for (int i = 0; i < 16; ++i) s += qs[16 * g + i];
            bsums[g] = (int16_t)s;
        }
        d = 1.0f / iscale;
    }
    memcpy(blk, &d, 4);
    memcpy(blk + 4, qs, QK);
    memcpy(blk + 260, bsums, 32);
}

void plm_ref_quantize_q8K(const float* x, uint8_t* xq, int64_t m, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t b = 0; b < nb; ++b)
            quantize_chunk(x + i * k + b * QK, xq + (i * nb + b) * Q8K_BYTES);
}

/* ------------------------------------------------------------------ */
/* q4_K: the 12-byte table of eight 6-bit (scale, min) pairs.          */
/* Pairs 0..3 sit in the low 6 bits of bytes 0..3 (scale) and 4..7     */
/* (min); pairs 4..7 take their low 4 bits from the nibbles of bytes   */
/* 8..11 and their top 2 bits from the spare top bits of bytes 0..7.   */
/* ------------------------------------------------------------------ */
void plm_ref_q4K_scale_min(const uint8_t* s, int j, int* sc, int* mn) {
    if (j < 4) {
        *sc = s[j] & 63;
        *mn = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* Sub-block dots of one q4_K block against one q8_K block.
 * dots[j] = sum_{l<32} q(32j+l) * q8(32j+l), j = 0..7.
 * Walks the 128 qs bytes: byte 32c+l holds weight 64c+l in its low nibble
 * (sub-block 2c) and weight 64c+32+l in its high nibble (sub-block 2c+1). */
static void q4K_block_dots(const uint8_t* wb, const int8_t* q8, int32_t dots[8]) {
    const uint8_t* qs = wb + 16;
    for (int j = 0; j < 8; ++j) dots[j] = 0;
    for (int c = 0; c < 4; ++c) {
        for (int l = 0; l < 32; ++l) {
            int byte = qs[32 * c + l];
            dots[2 * c]     += (byte & 15) * q8[64 * c + l];
            dots[2 * c + 1] += (byte >> 4) * q8[64 * c + 32 + l];
        }
    }
}

/* q6_K: six-bit code of every weight, from ql (low 4 bits) and qh (2 bits).
 * Half h (weights 128h..128h+127) uses ql[64h..64h+63] and qh[32h..32h+31];
 * for l < 32 the four quarters of the half are
 *   128h+l    : low  nibble of ql[64h+l],    qh bits 0-1 of qh[32h+l]
 *   128h+32+l : low  nibble of ql[64h+32+l], qh bits 2-3
 *   128h+64+l : high nibble of ql[64h+l],    qh bits 4-5
 *   128h+96+l : high nibble of ql[64h+32+l], qh bits 6-7              */
static void q6K_codes(const uint8_t* wb, int q[QK]) {
    const uint8_t* ql = wb;
    const uint8_t* qh = wb + 128;
    for (int h = 0; h < 2; ++h) {
        const uint8_t* L = ql + 64 * h;
        const uint8_t* H = qh + 32 * h;
        for (int l = 0; l < 32; ++l) {
            q[128 * h + l]      = (L[l] & 15)      | (((H[l] >> 0) & 3) << 4);
            q[128 * h + 32 + l] = (L[l + 32] & 15) | (((H[l] >> 2) & 3) << 4);
            q[128 * h + 64 + l] = (L[l] >> 4)      | (((H[l] >> 4) & 3) << 4);
            q[128 * h + 96 + l] = (L[l + 32] >> 4) | (((H[l] >> 6) & 3) << 4);
        }
    }
}

/* dots[g] = sum_{i<16} (q6(16g+i) - 32) * q8(16g+i), g = 0..15 */
static void q6K_block_dots(const uint8_t* wb, const int8_t* q8, int32_t dots[16]) {
    int q[QK];
    q6K_codes(wb, q);
    for (int g = 0; g < 16; ++g) {
        int32_t s = 0;
        for (int i = 0; i < 16; ++i) s += (q[16 * g + i] - 32) * q8[16 * g + i];
        dots[g] = s;
    }
}

/* ------------------------------------------------------------------ */
/* Exported integer sub-dots: out[i][r][b*8 + j] (q4_K), out[i][r][b*16 + g] (q6_K). */
/* ------------------------------------------------------------------ */
void plm_ref_subdots_q4K(const uint8_t* w, const uint8_t* xq, int32_t* out,
                         int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t r = 0; r < n; ++r)
            for (int64_t b = 0; b < nb; ++b)
                q4K_block_dots(w + (r * nb + b) * Q4K_BYTES,
                               (const int8_t*)(xq + (i * nb + b) * Q8K_BYTES + 4),
                               out + ((i * n + r) * nb + b) * 8);
}

void plm_ref_subdots_q6K(const uint8_t* w, const uint8_t* xq, int32_t* out,
                         int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t r = 0; r < n; ++r)
            for (int64_t b = 0; b < nb; ++b)
                q6K_block_dots(w + (r * nb + b) * Q6K_BYTES,
                               (const int8_t*)(xq + (i * nb + b) * Q8K_BYTES + 4),
                               out + ((i * n + r) * nb + b) * 16);
}

/* ------------------------------------------------------------------ */
/* Y = X . W^T through the integer path.                               */
/* Per block b of weight row r and activation row i:                   */
/*   q4_K: isum = sum_j sc_j*dot_j, msum = sum_j m_j*(bsum_2j+bsum_2j+1) */
/*         term = d_w*d_x*isum - dmin_w*d_x*msum                        */
/*   q6_K: isum = sum_g sc_g*dot_g, term = d_w*d_x*isum                */
/* Y[i][r] = sum of terms over b, in block order.                      */
/* ------------------------------------------------------------------ */
static void q4K_block_ints(const uint8_t* wb, const uint8_t* xb, int32_t* isum, int32_t* msum) {
    int32_t dots[8];
    q4K_block_dots(wb, (const int8_t*)(xb + 4), dots);
    int32_t is = 0, ms = 0;
    for (int j = 0; j < 8; ++j) {
        int sc, mn;
        plm_ref_q4K_scale_min(wb + 4, j, &sc, &mn);
        is += sc * dots[j];
        ms += mn * ((int32_t)load_i16(xb + 260 + 4 * j) + (int32_t)load_i16(xb + 260 + 4 * j + 2));
    }
    *isum = is;
    *msum = ms;
}

static int32_t q6K_block_ints(const uint8_t* wb, const uint8_t* xb) {
    int32_t dots[16];
    q6K_block_dots(wb, (const int8_t*)(xb + 4), dots);
    const int8_t* sc = (const int8_t*)(wb + 192);
    int32_t is = 0;
    for (int g = 0; g < 16; ++g) is += (int32_t)sc[g] * dots[g];
    return is;
}

void plm_ref_gemm_q4K_f64(const uint8_t* w, const uint8_t* xq, double* y,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q4K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                int32_t isum, msum;
                q4K_block_ints(wb, xb, &isum, &msum);
                double dx = (double)load_f32(xb);
                acc += (double)load_f16(wb) * dx * (double)isum
                     - (double)load_f16(wb + 2) * dx * (double)msum;
            }
            y[i * n + r] = acc;
        }
    }
}

void plm_ref_gemm_q4K_f32(const uint8_t* w, const uint8_t* xq, float* y,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            float acc = 0.0f;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q4K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                int32_t isum, msum;
                q4K_block_ints(wb, xb, &isum, &msum);
                float dx = load_f32(xb);
                acc += load_f16(wb) * dx * (float)isum - load_f16(wb + 2) * dx * (float)msum;
            }
            y[i * n + r] = acc;
        }
    }
}

void plm_ref_gemm_q6K_f64(const uint8_t* w, const uint8_t* xq, double* y,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q6K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                acc += (double)load_f16(wb + 208) * (double)load_f32(xb) * (double)q6K_block_ints(wb, xb);
            }
            y[i * n + r] = acc;
        }
    }
}

void plm_ref_gemm_q6K_f32(const uint8_t* w, const uint8_t* xq, float* y,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            float acc = 0.0f;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q6K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                acc += load_f16(wb + 208) * load_f32(xb) * (float)q6K_block_ints(wb, xb);
            }
            y[i * n + r] = acc;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Dequantization to f64, one weight at a time from its index.         */
/* Written per weight (not per byte) so that it checks the byte walks  */
/* of the integer path above from a second direction.                  */
/* ------------------------------------------------------------------ */
void plm_ref_dequant_q4K(const uint8_t* w, double* out, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* wb = w + (r * nb + b) * Q4K_BYTES;
            double d = load_f16(wb), dmin = load_f16(wb + 2);
            for (int t = 0; t < QK; ++t) {
                int chunk = t / 64, within = t % 64;
                int byte = wb[16 + 32 * chunk + within % 32];
                int q = within < 32 ? (byte & 15) : (byte >> 4);
                int sc, mn;
                plm_ref_q4K_scale_min(wb + 4, t / 32, &sc, &mn);
                out[r * k + b * QK + t] = d * sc * q - dmin * mn;
            }
        }
}

/* The row-interleaved q4_K layout "x16" (a repack of the same bytes for the
 * GPU decode GEMV, the analogue of the pages' panel repack of q4_K weights,
 * Korean README, "Current status" table, row "src/").  Definition: rows in
 * tiles of 16; the tile-block of tile T, block b is 2304 bytes at
 * (T*nb + b)*2304; its bytes 16i .. 16i+15 are the header (d, dmin,
 * scales[12]) of row 16T + i; for j = 0..3, L = 0..31 (g = L/4, t = L%4) its
 * bytes 256 + 512j + 16L .. +15 are qs[32t + 16(j%2) .. +15] of row 16T + g
 * (j < 2) or 16T + g + 8 (j >= 2).  Below: the inverse walk, from a row's
 * qs byte c to its place, then the q4_K decode of dequant_q4K. */
static const uint8_t* x16_qs_byte(const uint8_t* tb, int i, int c) {
    int t = c / 32, within = c % 32;
    int g = i % 8, j = (i < 8 ? 0 : 2) + within / 16;
    return tb + 256 + 512 * j + 16 * (4 * g + t) + within % 16;
}

void plm_ref_dequant_q4K_x16(const uint8_t* wx, double* out, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* tb = wx + ((r / 16) * nb + b) * (16 * Q4K_BYTES);
            const uint8_t* hdr = tb + 16 * (r % 16);
            double d = load_f16(hdr), dmin = load_f16(hdr + 2);
            for (int t = 0; t < QK; ++t) {
                int chunk = t / 64, within = t % 64;
                int byte = *x16_qs_byte(tb, (int)(r % 16), 32 * chunk + within % 32);
                int q = within < 32 ? (byte & 15) : (byte >> 4);
                int sc, mn;
                plm_ref_q4K_scale_min(hdr + 4, t / 32, &sc, &mn);
                out[r * k + b * QK + t] = d * sc * q - dmin * mn;
            }
        }
}

/* The x16 layout of q6_K: rows in tiles of 16; the tile-block of tile T,
 * block b is 3360 bytes at (T*nb + b)*3360: bytes 16i .. 16i+15 are the int8
 * scales of row 16T + i, bytes 256 + 2i .. +1 its f16 d; for j = 0..3 and
 * L = 0..31 (g = L/4, t = L%4), bytes 288 + 512j + 16L + 4w .. +3 (w = 0..3)
 * are ql[64(j%2) + 16w + 4t .. +3] of row 16T + g (j < 2) or 16T + g + 8;
 * for j = 0..1, bytes 2336 + 512j + 16L + 4p .. +3 (p = 2h + s) are
 * qh[32h + 16s + 4t .. +3] of row 16T + g + 8j.  Below: the inverse walk
 * from a row's ql / qh byte to its place, then the q6_K decode of
 * dequant_q6K. */
static const uint8_t* x16_q6K_ql(const uint8_t* tb, int i, int c) {   /* ql[c], c < 128 */
    int h = c / 64, w = (c % 64) / 16, t = (c % 16) / 4, e = c % 4;
    int g = i % 8, j = (i < 8 ? 0 : 2) + h;
    return tb + 288 + 512 * j + 16 * (4 * g + t) + 4 * w + e;
}
static const uint8_t* x16_q6K_qh(const uint8_t* tb, int i, int c) {   /* qh[c], c < 64 */
    int h = c / 32, s = (c % 32) / 16, t = (c % 16) / 4, e = c % 4;
    int g = i % 8, j = i < 8 ? 0 : 1;
    return tb + 2336 + 512 * j + 16 * (4 * g + t) + 4 * (2 * h + s) + e;
}

void plm_ref_dequant_q6K_x16(const uint8_t* wx, double* out, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* tb = wx + ((r / 16) * nb + b) * (16 * Q6K_BYTES);
            int i = (int)(r % 16);
            double d = load_f16(tb + 256 + 2 * i);
            for (int t = 0; t < QK; ++t) {
                int half = t / 128, quarter = (t % 128) / 32, l = t % 32;
                int lbyte = *x16_q6K_ql(tb, i, 64 * half + 32 * (quarter & 1) + l);
                int low4 = (quarter & 2) ? (lbyte >> 4) : (lbyte & 15);
                int high2 = (*x16_q6K_qh(tb, i, 32 * half + l) >> (2 * quarter)) & 3;
                int q = low4 | (high2 << 4);
                int sc = (int8_t)tb[16 * i + t / 16];
                out[r * k + b * QK + t] = d * sc * (q - 32);
            }
        }
}

void plm_ref_dequant_q6K(const uint8_t* w, double* out, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* wb = w + (r * nb + b) * Q6K_BYTES;
            double d = load_f16(wb + 208);
            for (int t = 0; t < QK; ++t) {
                int half = t / 128, quarter = (t % 128) / 32, l = t % 32;
                int lbyte = wb[64 * half + 32 * (quarter & 1) + l];
                int low4 = (quarter & 2) ? (lbyte >> 4) : (lbyte & 15);
                int high2 = (wb[128 + 32 * half + l] >> (2 * quarter)) & 3;
                int q = low4 | (high2 << 4);
                int sc = (int8_t)wb[192 + t / 16];
                out[r * k + b * QK + t] = d * sc * (q - 32);
            }
        }
}

void plm_ref_dequant_q8K(const uint8_t* xq, double* out, int64_t m, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
            double d = load_f32(xb);
            for (int t = 0; t < QK; ++t)
                out[i * k + b * QK + t] = d * (double)(int8_t)xb[4 + t];
        }
}

/* S[i][r] = sum over k of |w_hat * x_hat| in f64: the scale that the f32
 * tolerance is relative to. */
void plm_ref_absscale_q4K(const uint8_t* w, const uint8_t* xq, double* S,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        double wr[QK];
        for (int64_t i = 0; i < m; ++i) S[i * n + r] = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            plm_ref_dequant_q4K(w + (r * nb + b) * Q4K_BYTES, wr, 1, QK);
            for (int64_t i = 0; i < m; ++i) {
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                double dx = load_f32(xb), s = 0.0;
                for (int t = 0; t < QK; ++t) s += fabs(wr[t] * dx * (double)(int8_t)xb[4 + t]);
                S[i * n + r] += s;
            }
        }
    }
}

void plm_ref_absscale_q6K(const uint8_t* w, const uint8_t* xq, double* S,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        double wr[QK];
        for (int64_t i = 0; i < m; ++i) S[i * n + r] = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            plm_ref_dequant_q6K(w + (r * nb + b) * Q6K_BYTES, wr, 1, QK);
            for (int64_t i = 0; i < m; ++i) {
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                double dx = load_f32(xb), s = 0.0;
                for (int t = 0; t < QK; ++t) s += fabs(wr[t] * dx * (double)(int8_t)xb[4 + t]);
                S[i * n + r] += s;
            }
        }
    }
}

/* Thread control for the OpenMP row loops (1 = single-threaded). */
void plm_ref_set_threads(int t) {
#ifdef _OPENMP
    omp_set_num_threads(t > 0 ? t : 1);
#else
    (void)t;
#endif
}

int plm_ref_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Array form of the binary16 decode, for exhaustive host checks. */
void plm_ref_f16_array(const uint16_t* h, float* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = plm_ref_f16_to_f32(h[i]);
}

/*
 * SwiGLU epilogue of an ffn gate/up pair (PocketLLM, Korean README,
 * "Current status" table, row "src/": the decode path's silu_mul step):
 *   h = silu(g) * u,  silu(g) = g * sigmoid(g) = g / (1 + exp(-g)),
 * in f64, elementwise over count values.
 */
void plm_ref_swiglu_f64(const double* g, const double* u, double* h, int64_t count) {
    for (int64_t i = 0; i < count; ++i) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* ------------------------------------------------------------------ */
/* q5_K: the q4_K layout plus qh[32] (the fifth bit of every weight).  */
/* Byte 32c+l of qs and byte l of qh give weight 64c+l (low nibble,    */
/* qh bit 2c, sub-block 2c) and weight 64c+32+l (high nibble, qh bit   */
/* 2c+1, sub-block 2c+1).  The scale/min table is q4_K's.             */
/* ------------------------------------------------------------------ */
static void q5K_block_dots(const uint8_t* wb, const int8_t* q8, int32_t dots[8]) {
    const uint8_t* qh = wb + 16;
    const uint8_t* qs = wb + 48;
    for (int c = 0; c < 4; ++c) {
        int32_t lo = 0, hi = 0;
        for (int l = 0; l < 32; ++l) {
            int byte = qs[32 * c + l];
            int q0 = (byte & 15) + 16 * ((qh[l] >> (2 * c)) & 1);
            int q1 = (byte >> 4) + 16 * ((qh[l] >> (2 * c + 1)) & 1);
            lo += q0 * q8[64 * c + l];
            hi += q1 * q8[64 * c + 32 + l];
        }
        dots[2 * c] = lo;
        dots[2 * c + 1] = hi;
    }
}

static void q5K_block_ints(const uint8_t* wb, const uint8_t* xb, int32_t* isum, int32_t* msum) {
    int32_t dots[8];
    q5K_block_dots(wb, (const int8_t*)(xb + 4), dots);
    int32_t is = 0, ms = 0;
    for (int j = 0; j < 8; ++j) {
        int sc, mn;
        plm_ref_q4K_scale_min(wb + 4, j, &sc, &mn);
        is += sc * dots[j];
        ms += mn * ((int32_t)load_i16(xb + 260 + 4 * j) + (int32_t)load_i16(xb + 260 + 4 * j + 2));
    }
    *isum = is;
    *msum = ms;
}

void plm_ref_subdots_q5K(const uint8_t* w, const uint8_t* xq, int32_t* out,
                         int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t r = 0; r < n; ++r)
            for (int64_t b = 0; b < nb; ++b)
                q5K_block_dots(w + (r * nb + b) * Q5K_BYTES,
                               (const int8_t*)(xq + (i * nb + b) * Q8K_BYTES + 4),
                               out + ((i * n + r) * nb + b) * 8);
}

void plm_ref_gemm_q5K_f64(const uint8_t* w, const uint8_t* xq, double* y,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q5K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                int32_t isum, msum;
                q5K_block_ints(wb, xb, &isum, &msum);
                double dx = (double)load_f32(xb);
                acc += (double)load_f16(wb) * dx * (double)isum
                     - (double)load_f16(wb + 2) * dx * (double)msum;
            }
            y[i * n + r] = acc;
        }
    }
}

void plm_ref_gemm_q5K_f32(const uint8_t* w, const uint8_t* xq, float* y,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            float acc = 0.0f;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q5K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                int32_t isum, msum;
                q5K_block_ints(wb, xb, &isum, &msum);
                float dx = load_f32(xb);
                acc += load_f16(wb) * dx * (float)isum - load_f16(wb + 2) * dx * (float)msum;
            }
            y[i * n + r] = acc;
        }
    }
}

/* Per-weight f64 dequantization of q5_K (from the weight index). */
void plm_ref_dequant_q5K(const uint8_t* w, double* out, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* wb = w + (r * nb + b) * Q5K_BYTES;
            double d = load_f16(wb), dmin = load_f16(wb + 2);
            for (int t = 0; t < QK; ++t) {
                int chunk = t / 64, within = t % 64, l = within % 32, upper = within >= 32;
                int byte = wb[48 + 32 * chunk + l];
                int q = (upper ? (byte >> 4) : (byte & 15)) + 16 * ((wb[16 + l] >> (2 * chunk + upper)) & 1);
                int sc, mn;
                plm_ref_q4K_scale_min(wb + 4, t / 32, &sc, &mn);
                out[r * k + b * QK + t] = d * sc * q - dmin * mn;
            }
        }
}

void plm_ref_absscale_q5K(const uint8_t* w, const uint8_t* xq, double* S,
                          int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    double wr[QK];
    for (int64_t i = 0; i < m * n; ++i) S[i] = 0.0;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            plm_ref_dequant_q5K(w + (r * nb + b) * Q5K_BYTES, wr, 1, QK);
            for (int64_t i = 0; i < m; ++i) {
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                double dx = load_f32(xb), s = 0.0;
                for (int t = 0; t < QK; ++t) s += fabs(wr[t] * dx * (double)(int8_t)xb[4 + t]);
                S[i * n + r] += s;
            }
        }
}

/* ------------------------------------------------------------------ */
/* q2_K and q3_K (the lower rungs of the width ladder), public GGML    */
/* layouts.  Both use sixteen 16-weight groups; group g holds weights  */
/* 16g .. 16g+15 and, with h = g/8, j = (g%8)/2, p = g%2, its codes    */
/* sit in bits 2j, 2j+1 of qs[32h + 16p + l], l = 0..15.               */
/*   q2_K (84 B): u8 scales[16] (low nibble scale, high nibble min),   */
/*        u8 qs[64], f16 d, f16 dmin; weight = d*sc_g*q - dmin*m_g.    */
/*   q3_K (110 B): u8 hmask[32], u8 qs[64], u8 scales[12], f16 d; the  */
/*        third bit of weight 16g+l is bit 4h+j of hmask[16p+l]; code  */
/*        q3 = q2 - 4 when that bit is clear, else q2 (-4..3); the     */
/*        6-bit scale of group g takes its low 4 bits from             */
/*        scales[g%8] (nibble g/8) and its top 2 bits from bits        */
/*        2(g/4)..2(g/4)+1 of scales[8 + g%4]; weight = d*(s_g-32)*q3. */
/* ------------------------------------------------------------------ */
#define Q2K_BYTES 84
#define Q3K_BYTES 110

static int k2_code(const uint8_t* qs, int w) {
    int g = w / 16, l = w % 16, h = g / 8, j = (g % 8) / 2, p = g % 2;
    return (qs[32 * h + 16 * p + l] >> (2 * j)) & 3;
}

int plm_ref_q3K_scale(const uint8_t* sc12, int g) {
    int low4 = (sc12[g % 8] >> (4 * (g / 8))) & 15;
    int high2 = (sc12[8 + g % 4] >> (2 * (g / 4))) & 3;
    return low4 | (high2 << 4);
}

static int k3_code(const uint8_t* wb, int w) {
    int g = w / 16, l = w % 16, h = g / 8, j = (g % 8) / 2, p = g % 2;
    int hbit = (wb[16 * p + l] >> (4 * h + j)) & 1;
    return k2_code(wb + 32, w) - (hbit ? 0 : 4);
}

static void q2K_block_dots(const uint8_t* wb, const int8_t* q8, int32_t dots[16]) {
    for (int g = 0; g < 16; ++g) {
        int32_t s = 0;
        for (int l = 0; l < 16; ++l) s += k2_code(wb + 16, 16 * g + l) * q8[16 * g + l];
        dots[g] = s;
    }
}

static void q3K_block_dots(const uint8_t* wb, const int8_t* q8, int32_t dots[16]) {
    for (int g = 0; g < 16; ++g) {
        int32_t s = 0;
        for (int l = 0; l < 16; ++l) s += k3_code(wb, 16 * g + l) * q8[16 * g + l];
        dots[g] = s;
    }
}

void plm_ref_subdots_q2K(const uint8_t* w, const uint8_t* xq, int32_t* out, int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t r = 0; r < n; ++r)
            for (int64_t b = 0; b < nb; ++b)
                q2K_block_dots(w + (r * nb + b) * Q2K_BYTES, (const int8_t*)(xq + (i * nb + b) * Q8K_BYTES + 4),
                               out + ((i * n + r) * nb + b) * 16);
}

void plm_ref_subdots_q3K(const uint8_t* w, const uint8_t* xq, int32_t* out, int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t r = 0; r < n; ++r)
            for (int64_t b = 0; b < nb; ++b)
                q3K_block_dots(w + (r * nb + b) * Q3K_BYTES, (const int8_t*)(xq + (i * nb + b) * Q8K_BYTES + 4),
                               out + ((i * n + r) * nb + b) * 16);
}

/* Block integers: q2_K isum = sum_g sc_g dot_g, msum = sum_g m_g bsum_g;
 * q3_K isum = sum_g (s_g - 32) dot_g (no min term). */
static void q2K_block_ints(const uint8_t* wb, const uint8_t* xb, int32_t* isum, int32_t* msum) {
    int32_t dots[16];
    q2K_block_dots(wb, (const int8_t*)(xb + 4), dots);
    int32_t is = 0, ms = 0;
    for (int g = 0; g < 16; ++g) {
        is += (wb[g] & 15) * dots[g];
        ms += (wb[g] >> 4) * (int32_t)load_i16(xb + 260 + 2 * g);
    }
    *isum = is;
    *msum = ms;
}

static int32_t q3K_block_ints(const uint8_t* wb, const uint8_t* xb) {
    int32_t dots[16];
    q3K_block_dots(wb, (const int8_t*)(xb + 4), dots);
    int32_t is = 0;
    for (int g = 0; g < 16; ++g) is += (plm_ref_q3K_scale(wb + 96, g) - 32) * dots[g];
    return is;
}

void plm_ref_gemm_q2K_f64(const uint8_t* w, const uint8_t* xq, double* y, int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q2K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                int32_t isum, msum;
                q2K_block_ints(wb, xb, &isum, &msum);
                double dx = (double)load_f32(xb);
                acc += (double)load_f16(wb + 80) * dx * (double)isum - (double)load_f16(wb + 82) * dx * (double)msum;
            }
            y[i * n + r] = acc;
        }
}

void plm_ref_gemm_q2K_f32(const uint8_t* w, const uint8_t* xq, float* y, int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t i = 0; i < m; ++i) {
            float acc = 0.0f;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q2K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                int32_t isum, msum;
                q2K_block_ints(wb, xb, &isum, &msum);
                float dx = load_f32(xb);
                acc += load_f16(wb + 80) * dx * (float)isum - load_f16(wb + 82) * dx * (float)msum;
            }
            y[i * n + r] = acc;
        }
}

void plm_ref_gemm_q3K_f64(const uint8_t* w, const uint8_t* xq, double* y, int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q3K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                acc += (double)load_f16(wb + 108) * (double)load_f32(xb) * (double)q3K_block_ints(wb, xb);
            }
            y[i * n + r] = acc;
        }
}

void plm_ref_gemm_q3K_f32(const uint8_t* w, const uint8_t* xq, float* y, int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t i = 0; i < m; ++i) {
            float acc = 0.0f;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = w + (r * nb + b) * Q3K_BYTES;
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                acc += load_f16(wb + 108) * load_f32(xb) * (float)q3K_block_ints(wb, xb);
            }
            y[i * n + r] = acc;
        }
}

/* Per-weight f64 dequantization (from the weight index). */
void plm_ref_dequant_q2K(const uint8_t* w, double* out, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* wb = w + (r * nb + b) * Q2K_BYTES;
            double d = load_f16(wb + 80), dmin = load_f16(wb + 82);
            for (int t = 0; t < QK; ++t) {
                int sb = wb[t / 16];
                out[r * k + b * QK + t] = d * (sb & 15) * k2_code(wb + 16, t) - dmin * (sb >> 4);
            }
        }
}

void plm_ref_dequant_q3K(const uint8_t* w, double* out, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* wb = w + (r * nb + b) * Q3K_BYTES;
            double d = load_f16(wb + 108);
            for (int t = 0; t < QK; ++t)
                out[r * k + b * QK + t] = d * (plm_ref_q3K_scale(wb + 96, t / 16) - 32) * k3_code(wb, t);
        }
}

static void absscale_generic(void (*deq)(const uint8_t*, double*, int64_t, int64_t), int bpb, const uint8_t* w,
                             const uint8_t* xq, double* S, int64_t m, int64_t n, int64_t k) {
    int64_t nb = k / QK;
    double wr[QK];
    for (int64_t i = 0; i < m * n; ++i) S[i] = 0.0;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            deq(w + (r * nb + b) * bpb, wr, 1, QK);
            for (int64_t i = 0; i < m; ++i) {
                const uint8_t* xb = xq + (i * nb + b) * Q8K_BYTES;
                double dx = load_f32(xb), s = 0.0;
                for (int t = 0; t < QK; ++t) s += fabs(wr[t] * dx * (double)(int8_t)xb[4 + t]);
                S[i * n + r] += s;
            }
        }
}

void plm_ref_absscale_q2K(const uint8_t* w, const uint8_t* xq, double* S, int64_t m, int64_t n, int64_t k) {
    absscale_generic(plm_ref_dequant_q2K, Q2K_BYTES, w, xq, S, m, n, k);
}

void plm_ref_absscale_q3K(const uint8_t* w, const uint8_t* xq, double* S, int64_t m, int64_t n, int64_t k) {
    absscale_generic(plm_ref_dequant_q3K, Q3K_BYTES, w, xq, S, m, n, k);
}
