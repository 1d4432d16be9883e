/*
 * Seeded synthetic inputs for the packed-weight matmul (gemm_quant) of the
 * PocketLLM pages: q4_K and q6_K weight blocks and f32 activations.
 *
 * This file holds no arithmetic of the method itself.  It only fills the
 * block fields with random values of the distributions the workloads name:
 *   q4_K : d, dmin ~ U(1e-4, 2e-3) rounded to f16; the 12 scale bytes and the
 *          128 nibble bytes uniform.  Every 12-byte string is the packing of
 *          eight 6-bit (scale, min) pairs and the packing is a bijection on
 *          96 bits, so uniform bytes give scales and mins i.i.d. U{0..63};
 *          likewise uniform qs bytes give nibbles i.i.d. U{0..15}.
 *   q5_K : as q4_K, plus 32 uniform qh bytes (the fifth bit of each weight),
 *          so q5 ~ U{0..31}.
 *   q2_K : d, dmin as q4_K; scales[16] and qs[64] uniform bytes (4-bit scales
 *          and mins ~ U{0..15}, 2-bit codes ~ U{0..3}).
 *   q3_K : d as q4_K; hmask[32], qs[64] and scales[12] uniform bytes (3-bit
 *          codes ~ U{0..7} before the offset, 6-bit scales ~ U{0..63}).
 *   q6_K : d ~ U(1e-4, 2e-3) rounded to f16; ql[128] and qh[64] uniform bytes
 *          (a bijection onto 256 six-bit values, so q6 ~ U{0..63});
 *          scales i8 ~ U{-64..63}.
 *   x    : f32 ~ N(0,1) by Box-Muller in f64, cast to f32.
 *
 * Random numbers: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), used in its counter form:
 * draw i of a stream with start state s is mix(s + (i+1)*gamma), which is the
 * i-th output of the stateful generator started at s.  So any slice of a
 * tensor is generated on its own, in any order, with the same bytes.
 *
 * Stream start state: s = seed ^ (stream * 0xD1B54A32D192ED03).
 * Draw layout, per block index b of a stream:
 *   q4_K: 20 draws from 20*b.  draw 0 -> d, draw 1 -> dmin, draws 2..19 give
 *         8 bytes each (little-endian) for scales[12] then qs[128]
 *         (140 bytes used, 4 dropped).
 *   q2_K: 12 draws from 12*b.  draw 0 -> d, draw 1 -> dmin, draws 2..11 give
 *         scales[16] then qs[64].
 *   q3_K: 15 draws from 15*b.  draw 0 -> d, draws 1..14 give hmask[32],
 *         qs[64] then scales[12].
 *   q5_K: 24 draws from 24*b.  draw 0 -> d, draw 1 -> dmin, draws 2..23 give
 *         8 bytes each for scales[12], qh[32] then qs[128] (172 bytes used).
 *   q6_K: 27 draws from 27*b.  draw 0 -> d, draws 1..24 give ql[128] then
 *         qh[64], draws 25..26 give 16 bytes b, scale = (b & 127) - 64.
 *   x   : element e takes draws 2e (u1) and 2e+1 (u2).
 * Uniform in [0,1): (draw >> 11) * 2^-53.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t stream_start(uint64_t seed, uint64_t stream) {
    return seed ^ (stream * 0xD1B54A32D192ED03ULL);
}

static uint64_t draw(uint64_t s, uint64_t i) { return mix64(s + (i + 1) * GAMMA); }

static double unit(uint64_t r) { return (double)(r >> 11) * (1.0 / 9007199254740992.0); }

/* Round a positive normal-range double to IEEE binary16, nearest-even.
 * Only used for block scales in [1e-4, 2e-3], all normal halves. */
static uint16_t to_half_bits(double v) {
    int e;
    double f = frexp(v, &e);          /* v = f * 2^e, f in [0.5, 1) */
    /* half normal: v = (1 + mant/1024) * 2^(e-1), biased exponent e-1+15 */
    double scaled = f * 2048.0;       /* in [1024, 2048) */
    double fl = floor(scaled);
    double rem = scaled - fl;
    uint32_t sig = (uint32_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (sig & 1u))) sig += 1;
    int be = e - 1 + 15;
    if (sig == 2048) { sig = 1024; be += 1; }
    return (uint16_t)(((uint32_t)be << 10) | (sig - 1024));
}

static uint16_t draw_scale_half(uint64_t r) {
    double u = unit(r);
    return to_half_bits(1e-4 + u * (2e-3 - 1e-4));
}

static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

static void bytes_from_draws(uint64_t s, uint64_t first, uint8_t* out, int count) {
    for (int i = 0; i < count; ++i) {
        uint64_t r = draw(s, first + (uint64_t)(i / 8));
        out[i] = (uint8_t)((r >> (8 * (i % 8))) & 0xFF);
    }
}

void plmgen_q4K(uint64_t seed, uint64_t stream, int64_t block0, int64_t nblocks, uint8_t* out) {
    uint64_t s = stream_start(seed, stream);
    for (int64_t b = 0; b < nblocks; ++b) {
        uint64_t base = (uint64_t)(block0 + b) * 20u;
        uint8_t* blk = out + b * 144;
        uint8_t raw[144];
        put_u16(blk + 0, draw_scale_half(draw(s, base + 0)));
        put_u16(blk + 2, draw_scale_half(draw(s, base + 1)));
        bytes_from_draws(s, base + 2, raw, 140);
        memcpy(blk + 4, raw, 140);
    }
}

void plmgen_q2K(uint64_t seed, uint64_t stream, int64_t block0, int64_t nblocks, uint8_t* out) {
    uint64_t s = stream_start(seed, stream);
    for (int64_t b = 0; b < nblocks; ++b) {
        uint64_t base = (uint64_t)(block0 + b) * 12u;
        uint8_t* blk = out + b * 84;
        bytes_from_draws(s, base + 2, blk, 80);               /* scales[16], qs[64] */
        put_u16(blk + 80, draw_scale_half(draw(s, base + 0)));
        put_u16(blk + 82, draw_scale_half(draw(s, base + 1)));
    }
}

void plmgen_q3K(uint64_t seed, uint64_t stream, int64_t block0, int64_t nblocks, uint8_t* out) {
    uint64_t s = stream_start(seed, stream);
    for (int64_t b = 0; b < nblocks; ++b) {
        uint64_t base = (uint64_t)(block0 + b) * 15u;
        uint8_t* blk = out + b * 110;
        bytes_from_draws(s, base + 1, blk, 108);              /* hmask[32], qs[64], scales[12] */
        put_u16(blk + 108, draw_scale_half(draw(s, base + 0)));
    }
}

void plmgen_q5K(uint64_t seed, uint64_t stream, int64_t block0, int64_t nblocks, uint8_t* out) {
    uint64_t s = stream_start(seed, stream);
    for (int64_t b = 0; b < nblocks; ++b) {
        uint64_t base = (uint64_t)(block0 + b) * 24u;
        uint8_t* blk = out + b * 176;
        put_u16(blk + 0, draw_scale_half(draw(s, base + 0)));
        put_u16(blk + 2, draw_scale_half(draw(s, base + 1)));
        bytes_from_draws(s, base + 2, blk + 4, 172);
    }
}

void plmgen_q6K(uint64_t seed, uint64_t stream, int64_t block0, int64_t nblocks, uint8_t* out) {
    uint64_t s = stream_start(seed, stream);
    for (int64_t b = 0; b < nblocks; ++b) {
        uint64_t base = (uint64_t)(block0 + b) * 27u;
        uint8_t* blk = out + b * 210;
        uint8_t sb[16];
        bytes_from_draws(s, base + 1, blk, 192);            /* ql[128], qh[64] */
        bytes_from_draws(s, base + 25, sb, 16);
        for (int i = 0; i < 16; ++i) {
            int v = (int)(sb[i] & 127) - 64;
            blk[192 + i] = (uint8_t)(v & 0xFF);
        }
        put_u16(blk + 208, draw_scale_half(draw(s, base + 0)));
    }
}

void plmgen_normal_f32(uint64_t seed, uint64_t stream, int64_t elem0, int64_t count, float* out) {
    uint64_t s = stream_start(seed, stream);
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t e = 0; e < count; ++e) {
        uint64_t i = (uint64_t)(elem0 + e) * 2u;
        double u1 = 1.0 - unit(draw(s, i));     /* (0, 1] */
        double u2 = unit(draw(s, i + 1));
        double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        out[e] = (float)z;
    }
}

/* Raw draws, exposed so the host test can check the stream against the
 * published SplitMix64 sequence. */
void plmgen_raw(uint64_t seed, uint64_t stream, int64_t first, int64_t count, uint64_t* out) {
    uint64_t s = stream_start(seed, stream);
    for (int64_t i = 0; i < count; ++i) out[i] = draw(s, (uint64_t)(first + i));
}
