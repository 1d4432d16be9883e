// Decode GEMV, one lane per 256-weight block: q4_K and q5_K always, q2_K,
// q3_K and q6_K when a row's blocks keep every stage copy on 16-byte
// boundaries (lane_eligible, at the end) (PocketLLM "What it runs": K-quant
// weights decoded inside the kernel and never widened; the weight stream is
// read once for all m <= 8 activation rows, as the pages' 8-row activation
// tile does on the CPU).
//
// Work split: the weight stream of all problems of a launch is cut into
// row-aligned units (one stage each when a row has at most 32 blocks, else
// one row of several stages), and the units are split evenly over every
// warp of a persistent grid (one CTA per SM); a warp's range may run across
// problem boundaries.  Each warp streams its stages through a private ring
// of 32-block stages filled by bulk copies with bounded mbarrier waits.
//
// One warp step consumes one stage: lane L decodes block L of the stage in
// full (scales, mins, all eight 32-weight sub-blocks) against every
// activation row, so per-block fixed work is done once, not four times, and
// the cross-lane reduction is paid once per 32 blocks.  A stage holds
// floor(32 / nb) whole rows when nb <= 32 (row r on lanes [r*nb, r*nb+nb)),
// else 32 blocks of one row.  Row sums: butterfly over nb lanes when nb is a
// power of two, else a segmented shuffle-down; a row spanning several stages
// accumulates per lane first.  The f32 order of a row depends only on nb, so
// activation row i gives the same bits for every m and every grouping.
//
// Activations are staged once per CTA in shared memory, re-laid out per
// (row, block): the 256 codes, then the eight sums of adjacent bsum pairs
// (the min term's operands), 272 bytes apart so that eight lanes reading
// eight different blocks at the same offset hit distinct banks; the scales d
// sit in a separate float array, all at kernel start.
//
// XF32 (the fused q8_K producer): the problems carry f32 activations and the
// CTA quantizes them itself while staging (q8K_quantize_warp, the same
// arithmetic as the stand-alone quantizer), so the staged records and every
// output bit equal those of quantize + GEMV, without the q8_K round trip
// through memory or the second launch.
#pragma once

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "gemv_impl.cuh"

namespace plm {
namespace q4lane {

constexpr int STAGE_BLOCKS = 32;
// Staged bytes per activation block: the 256 codes, then q4_K/q5_K the eight
// sums of adjacent bsum pairs (272 bytes, a stride of 68 words), q2_K, q3_K
// and q6_K the sixteen bsums (304 bytes, 76 words); either way eight lanes
// reading eight different blocks at one offset hit distinct banks.
template <int FMT> __host__ __device__ constexpr int rec_bytes() { return FMT == 4 || FMT == 5 ? 272 : 304; }

// Block formats of this kernel: q4_K and q5_K (q4_K plus qh[32], the fifth
// bit of every weight, between the scale table and qs), whole 16-byte
// multiples, so every block of a stage is 16-byte aligned; q2_K (84 bytes:
// scales[16], qs[64], f16 d, f16 dmin), whose blocks are 4-byte aligned in a
// stage; q3_K (110 bytes: hmask[32], qs[64], scales[12], f16 d) and q6_K
// (210 bytes: ql[128], qh[64], int8 scales[16], f16 d), whose blocks sit at
// even offsets.  Their stages are 16-byte multiples starting on 16-byte
// boundaries when a row holds a multiple of four (q2_K: 4 * 84 = 21 * 16) or
// eight blocks (q3_K: 8 * 110 = 55 * 16; q6_K: 8 * 210 = 105 * 16), which
// the host requires of these formats on this kernel.
template <int FMT> struct LaneFmt;
template <> struct LaneFmt<4> {
    static constexpr int BYTES = Q4K_BYTES;
    static constexpr int QS = 16;                            // offset of qs[128]
};
template <> struct LaneFmt<5> {
    static constexpr int BYTES = Q5K_BYTES;
    static constexpr int QS = 48;
};
template <> struct LaneFmt<6> {
    static constexpr int BYTES = Q6K_BYTES;
    static constexpr int QS = 0;
};
template <> struct LaneFmt<2> {
    static constexpr int BYTES = Q2K_BYTES;
    static constexpr int QS = 16;
};
template <> struct LaneFmt<3> {
    static constexpr int BYTES = Q3K_BYTES;
    static constexpr int QS = 32;
};
// integer sub-block dots per block in the verification export
template <int FMT> __host__ __device__ constexpr int sub_per_block() { return FMT == 4 || FMT == 5 ? 8 : 16; }
template <int FMT> __host__ __device__ constexpr int slot_bytes() { return STAGE_BLOCKS * LaneFmt<FMT>::BYTES; }

// Bytes of one staged segment of nblk activation blocks: records, then the
// scales, padded to 16 bytes so the next segment's records stay aligned.
template <int FMT>
__host__ __device__ __forceinline__ int seg_bytes(int nblk) { return nblk * rec_bytes<FMT>() + ((nblk * 4 + 15) & ~15); }

// One problem of a launch.  Work is cut into units: rps whole rows (one
// stage) when a row has at most 32 blocks, else one row (ceil(nb / 32)
// stages, weight ceil(nb / 32)).  wbegin is the problem's first unit in the
// launch's weighted unit space.
struct LaneProblem {
    const uint8_t* w;
    const uint8_t* xq;
    float* y;
    int32_t* sub;
    int n, nb;
    int rps;                // rows per unit (0: one row per unit, several stages)
    int wbegin;             // weighted units before this problem
    const uint8_t* w2;      // paired launches: the up matrix (w is the gate matrix)
};

template <int MAXP>
struct LaneBatch {
    unsigned* fault;
    int count;
    int nstages;            // ring depth per warp
    int act_bytes;          // staged-activation region (all problems of the CTA)
    int wtotal;             // weighted units of the launch
    int prefetch;           // copy weights before waiting for the kernels before this one
    LaneProblem p[MAXP];
};

__host__ __device__ __forceinline__ int unit_weight(int nb) { return nb <= STAGE_BLOCKS ? 1 : (nb + STAGE_BLOCKS - 1) / STAGE_BLOCKS; }
__host__ __device__ __forceinline__ int unit_count(int n, int rps) { return rps > 0 ? (n + rps - 1) / rps : n; }
// Stages of one unit: a paired launch streams the gate rows, then the same up rows.
__host__ __device__ __forceinline__ int unit_stages(int nb, int pairf) { return unit_weight(nb) * pairf; }

// A warp's position in its unit range: problem p, unit u of [u, uend), chunk ch
// of the unit's row (one-row units only).  p < 0: the range is exhausted.
struct Cursor {
    int p, u, uend, ch;
};

// Moves to the first problem at or after p that has a unit starting in [W0, W1).
template <int MAXP>
__device__ __forceinline__ void cursor_enter(const LaneBatch<MAXP>& B, Cursor& c, int p, int W0, int W1, int pairf) {
    for (; p < B.count && B.p[p].wbegin < W1; ++p) {
        const LaneProblem& P = B.p[p];
        const int wt = unit_stages(P.nb, pairf);
        const int a = W0 - P.wbegin, b = W1 - P.wbegin;
        const int u0 = a > 0 ? (a + wt - 1) / wt : 0;
        const int u1 = min(unit_count(P.n, P.rps), (b + wt - 1) / wt);
        if (u0 < u1) {
            c = Cursor{p, u0, u1, 0};
            return;
        }
    }
    c.p = -1;
}

template <int MAXP>
__device__ __forceinline__ void cursor_next(const LaneBatch<MAXP>& B, Cursor& c, int nb, int W0, int W1, int pairf) {
    if (++c.ch < unit_stages(nb, pairf)) return;
    c.ch = 0;
    if (++c.u < c.uend) return;
    cursor_enter(B, c, c.p + 1, W0, W1, pairf);
}

// First block (within the row) of one-row stage ch; paired launches run the
// up matrix's stages after the gate's.
__device__ __forceinline__ int stage_b0(int ch, int nb) {
    const int spr = unit_weight(nb);
    return (ch >= spr ? ch - spr : ch) * STAGE_BLOCKS;
}

// SwiGLU epilogue of a paired launch: silu(g) * u = g / (1 + e^-g) * u.
__device__ __forceinline__ float swiglu(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// Last problem whose weighted range starts at or before W.
template <int MAXP>
__device__ __forceinline__ int problem_at(const LaneBatch<MAXP>& B, int W) {
    int r = 0;
    for (int lo = 1, hi = B.count - 1; lo <= hi;) {
        const int mid = (lo + hi) >> 1;
        if (B.p[mid].wbegin <= W) { r = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    return r;
}

// Activation staging.  A CTA stages the activations of every problem its
// warps touch, problems [p0, pend) of the launch, one segment per problem in
// launch order: m * nb records of REC bytes (the 256 codes, then the eight
// int16 sums of adjacent bsums), then the m * nb scales d as floats.  The
// first loads of a thread are issued before its warp fills the weight ring
// (fill()), so they are not queued behind the first weight stages of every
// SM; the staging then completes while those stages are in flight.

// Walks a flat index over the concatenated problems [p, pend): problem p
// covers [lo, hi) and its segment starts off bytes into the staging area.
struct ActPos {
    int p, lo, hi, off;
};
template <int M, int PER, int MAXP>
__device__ __forceinline__ ActPos act_begin(const LaneBatch<MAXP>& B, int p0, int pend) {
    return ActPos{p0, 0, p0 < pend ? M * B.p[p0].nb * PER : 0, 0};
}
template <int FMT, int M, int PER, int MAXP>
__device__ __forceinline__ void act_seek(const LaneBatch<MAXP>& B, ActPos& a, int idx, int pend) {
    while (a.p < pend && idx >= a.hi) {
        a.off += seg_bytes<FMT>(M * B.p[a.p].nb);
        a.lo = a.hi;
        ++a.p;
        a.hi = a.p < pend ? a.lo + M * B.p[a.p].nb * PER : a.lo;
    }
}

// Word w of a problem's q8_K rows (records of 73 words: d, 64 code words,
// 8 words of bsum pairs) into its staged segment of nblk records.
template <int FMT>
__device__ __forceinline__ void act_store(uint8_t* seg, int nblk, int w, uint32_t v) {
    constexpr int WORDS = Q8K_BYTES / 4;
    constexpr int REC = rec_bytes<FMT>();
    const int blk = w / WORDS;
    const int wd = w - blk * WORDS;
    if (wd == 0) {
        reinterpret_cast<float*>(seg + (size_t)nblk * REC)[blk] = __uint_as_float(v);
    } else if (wd <= 64) {
        reinterpret_cast<uint32_t*>(seg + (size_t)blk * REC)[wd - 1] = v;
    } else if constexpr (FMT != 4 && FMT != 5) {
        reinterpret_cast<uint32_t*>(seg + (size_t)blk * REC + 256)[wd - 65] = v;   // bsums 2j, 2j+1 as they are
    } else {
        const int j = wd - 65;   // bsums 2j, 2j+1
        const int pair = (int)(int16_t)(v & 0xFFFFu) + (int)(int16_t)(v >> 16);
        reinterpret_cast<int16_t*>(seg + (size_t)blk * REC + 256)[j] = (int16_t)pair;
    }
}

// q8_K activations: all threads of the CTA copy words, PRE of them per thread
// loaded before fill().
template <int FMT, int M, int PRE, int MAXP, typename Fill>
__device__ __forceinline__ void stage_q8(const LaneBatch<MAXP>& B, int p0, int pend, uint8_t* smem, Fill fill) {
    constexpr int WORDS = Q8K_BYTES / 4;
    const int tid = threadIdx.x, bd = blockDim.x;
    uint32_t pre[PRE];
    ActPos a = act_begin<M, WORDS>(B, p0, pend);
#pragma unroll
    for (int j = 0; j < PRE; ++j) {
        const int idx = tid + j * bd;
        act_seek<FMT, M, WORDS>(B, a, idx, pend);
        pre[j] = a.p < pend ? __ldg(reinterpret_cast<const uint32_t*>(B.p[a.p].xq) + (idx - a.lo)) : 0u;
    }
    fill();
    a = act_begin<M, WORDS>(B, p0, pend);
#pragma unroll
    for (int j = 0; j < PRE; ++j) {
        const int idx = tid + j * bd;
        act_seek<FMT, M, WORDS>(B, a, idx, pend);
        if (a.p < pend) act_store<FMT>(smem + a.off, M * B.p[a.p].nb, idx - a.lo, pre[j]);
    }
    for (int idx = tid + PRE * bd;; idx += bd) {
        act_seek<FMT, M, WORDS>(B, a, idx, pend);
        if (a.p >= pend) break;
        act_store<FMT>(smem + a.off, M * B.p[a.p].nb, idx - a.lo,
                       __ldg(reinterpret_cast<const uint32_t*>(B.p[a.p].xq) + (idx - a.lo)));
    }
}

// f32 activations (the fused producer): the CTA quantizes each 256-value
// chunk straight into the staged layout, one warp per chunk, the warps
// taking the chunks of all its problems in turn (chunk c of a problem's m
// rows starts at x + 256 c); a warp's first chunk is loaded before fill().
template <int M, int WARPS, int MAXP, typename Fill>
__device__ __forceinline__ void stage_f32(const LaneBatch<MAXP>& B, int p0, int pend, uint8_t* smem, int warp,
                                          int lane, Fill fill) {
    constexpr int REC = rec_bytes<4>();
    ActPos a = act_begin<M, 1>(B, p0, pend);
    int fc = warp;
    act_seek<4, M, 1>(B, a, fc, pend);
    float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
    if (a.p < pend) {
        const float4* src = reinterpret_cast<const float4*>(B.p[a.p].xq) + (size_t)(fc - a.lo) * (QK / 4) + 2 * lane;
        v0 = __ldg(src);
        v1 = __ldg(src + 1);
    }
    fill();
    while (a.p < pend) {
        const int nblk = M * B.p[a.p].nb;
        const int c = fc - a.lo;
        uint8_t* seg = smem + a.off;
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        int q[8];
        const float d = q8K_quantize_warp(v, lane, q);
        uint32_t w0, w1;
        pack_codes8(q, w0, w1);
        uint32_t* dst = reinterpret_cast<uint32_t*>(seg + (size_t)c * REC) + 2 * lane;
        dst[0] = w0;
        dst[1] = w1;
        // lanes 4j .. 4j+3 hold values 32j .. 32j+31: the sum of bsums 2j and 2j+1
        int sq = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
        sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 1);
        sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 2);
        if ((lane & 3) == 0) reinterpret_cast<int16_t*>(seg + (size_t)c * REC + 256)[lane >> 2] = (int16_t)sq;
        if (lane == 0) reinterpret_cast<float*>(seg + (size_t)nblk * REC)[c] = d;
        fc += WARPS;
        act_seek<4, M, 1>(B, a, fc, pend);
        if (a.p < pend) {
            const float4* src =
                reinterpret_cast<const float4*>(B.p[a.p].xq) + (size_t)(fc - a.lo) * (QK / 4) + 2 * lane;
            v0 = __ldg(src);
            v1 = __ldg(src + 1);
        }
    }
}

__device__ __forceinline__ int dp2a_hi_su(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// signed 16-bit halves of a times signed bytes 0, 1 of b
__device__ __forceinline__ int dp2a_lo_ss(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// One whole q4_K block against M staged activation blocks (same column,
// records act_stride bytes apart, scales dy_stride floats apart).  Adds the
// block's f32 term to v[i], or writes the eight exact sub-block dots.
// A block's 16-byte words, read from the stage in shared memory or from a
// copy the lane already holds in registers.
struct SmemBlock {
    const uint8_t* p;
    __device__ __forceinline__ uint4 at(int i) const { return reinterpret_cast<const uint4*>(p)[i]; }
};
template <int N>
struct RegBlock {
    uint4 r[N];
    __device__ __forceinline__ uint4 at(int i) const { return r[i]; }
};

template <int FMT, int M, bool SUBDOTS, class Blk>
__device__ __forceinline__ void lane_block(const Blk& w, const uint8_t* act, int act_stride, const float* dy,
                                           int dy_stride, float* v, int32_t* sub, size_t sub_stride) {
    const uint4 hdr = w.at(0);
    uint32_t qh[8];   // q5_K: the fifth bits, byte l <-> byte l of every qs chunk
    if constexpr (FMT == 5) {
        const uint4 h0 = w.at(1), h1 = w.at(2);
        qh[0] = h0.x; qh[1] = h0.y; qh[2] = h0.z; qh[3] = h0.w;
        qh[4] = h1.x; qh[5] = h1.y; qh[6] = h1.z; qh[7] = h1.w;
    }
    // six-bit scales (sc) and mins (m) as bytes: j = 0..3 and j = 4..7
    const uint32_t scA = hdr.y & 0x3F3F3F3Fu;
    const uint32_t mA = hdr.z & 0x3F3F3F3Fu;
    const uint32_t scB = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t mB = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    int isum[M];
#pragma unroll
    for (int i = 0; i < M; ++i) isum[i] = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 qa = w.at(LaneFmt<FMT>::QS / 16 + 2 * c);
        const uint4 qb = w.at(LaneFmt<FMT>::QS / 16 + 2 * c + 1);
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        // the codes of sub-blocks 2c (lo) and 2c+1 (hi) as bytes; q4_K's high
        // nibbles stay in place (16 q), divided out of the dot below
        uint32_t cl[8], ch[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if constexpr (FMT == 5) {
                cl[u] = (q[u] & 0x0F0F0F0Fu) | (((qh[u] >> (2 * c)) & 0x01010101u) << 4);
                ch[u] = ((q[u] >> 4) & 0x0F0F0F0Fu) | (((qh[u] >> (2 * c + 1)) & 0x01010101u) << 4);
            } else {
                cl[u] = q[u] & 0x0F0F0F0Fu;
                ch[u] = q[u] & 0xF0F0F0F0u;
            }
        }
        const uint32_t sw = c < 2 ? scA : scB;
        const int s0 = (int)((sw >> (16 * (c & 1))) & 0xFFu);
        const int s1 = (int)((sw >> (16 * (c & 1) + 8)) & 0xFFu);
#pragma unroll
        for (int i = 0; i < M; ++i) {
            const int4* x = reinterpret_cast<const int4*>(act + (size_t)i * act_stride + 64 * c);
            const int4 x0 = x[0], x1 = x[1], x2 = x[2], x3 = x[3];
            const int xl[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const int xh[8] = {x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
            int lo = 0, hi = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                lo = dp4a_us(cl[u], xl[u], lo);
                hi = dp4a_us(ch[u], xh[u], hi);
            }
            if constexpr (FMT == 4) hi >>= 4;   // the high nibbles were used in place (16 * q)
            if constexpr (SUBDOTS) {
                sub[i * sub_stride + 2 * c] = lo;
                sub[i * sub_stride + 2 * c + 1] = hi;
            } else {
                isum[i] += s0 * lo + s1 * hi;
            }
        }
    }
    if constexpr (!SUBDOTS) {
        const float d = half_bits_to_float(hdr.x);
        const float dmin = half_bits_to_float(hdr.x >> 16);
#pragma unroll
        for (int i = 0; i < M; ++i) {
            const int4 pr = *reinterpret_cast<const int4*>(act + (size_t)i * act_stride + 256);
            int ms = dp2a_lo_su(pr.x, mA, 0);
            ms = dp2a_hi_su(pr.y, mA, ms);
            ms = dp2a_lo_su(pr.z, mB, ms);
            ms = dp2a_hi_su(pr.w, mB, ms);
            const float tt = __fmaf_rn(d, (float)isum[i], -__fmul_rn(dmin, (float)ms));
            v[i] = __fmaf_rn(dy[i * dy_stride], tt, v[i]);
        }
    }
}

// q2_K, q3_K, q6_K: a block as four-byte words, read into registers.
// q2_K (4-byte aligned): all 21 words.  q3_K and q6_K sit at even offsets
// of the stage: their first 108 (27 words: hmask, qs, scales) and 208 bytes
// (52 words: ql, qh, scales) are read from the 4-byte boundary at or below
// the block and, for a block at 2 mod 4, realigned by a byte permute (bytes
// 2, 3 of one word, 0, 1 of the next); d has its own 2-byte load.  The NW + 1
// words read end with the block's last byte for a block at 2 mod 4, and two
// bytes past it for a block at 0 mod 4, which is never the last of a full
// slot (the 32nd block of 110- or 210-byte blocks sits at 2 mod 4): every
// load stays inside the stage slot.
template <int FMT> struct WordBlock;
template <> struct WordBlock<2> { static constexpr int NW = 21; uint32_t w[NW]; uint32_t d; };
template <> struct WordBlock<3> { static constexpr int NW = 27; uint32_t w[NW]; uint32_t d; };
template <> struct WordBlock<6> { static constexpr int NW = 52; uint32_t w[NW]; uint32_t d; };
using Q6Block = WordBlock<6>;

template <int FMT>
__device__ __forceinline__ void word_block_load(const uint8_t* blk, WordBlock<FMT>& B) {
    constexpr int NW = WordBlock<FMT>::NW;
    if constexpr (FMT == 2) {
        const uint32_t* p = reinterpret_cast<const uint32_t*>(blk);
#pragma unroll
        for (int j = 0; j < NW; ++j) B.w[j] = p[j];
        B.d = 0u;   // d, dmin are word 20
    } else {
        const uint32_t mis = (uint32_t)(uintptr_t)blk & 2u;
        const uint32_t* p = reinterpret_cast<const uint32_t*>(blk - mis);
        const uint32_t sel = mis ? 0x5432u : 0x3210u;
        uint32_t prev = p[0];
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const uint32_t next = p[j + 1];
            B.w[j] = __byte_perm(prev, next, sel);
            prev = next;
        }
        B.d = *reinterpret_cast<const uint16_t*>(blk + LaneFmt<FMT>::BYTES - 2);
    }
}

// One whole q6_K block against M staged activation blocks (records
// act_stride bytes apart: 256 codes, then the 16 bsums; scales dy_stride
// floats apart).  Weight 128h + 32qq + l takes its low four bits from
// ql[64h + 32(qq % 2) + l] (the low nibble for qq < 2) and its top two from
// bits 2qq, 2qq + 1 of qh[32h + l]; both are assembled four codes to a word
// and dotted with dp4a, and (q6 - 32) . x = q6 . x - 32 bsum per 16-weight
// group, exact in int32.  isum = sum of scale * group dot, exact in int32;
// then one f32 term per block, or the sixteen exact group dots.
template <int M, bool SUBDOTS>
__device__ __forceinline__ void lane_block_q6(const Q6Block& B, const uint8_t* act, int act_stride, const float* dy,
                                              int dy_stride, float* v, int32_t* sub, size_t sub_stride) {
    int isum[M];
#pragma unroll
    for (int i = 0; i < M; ++i) isum[i] = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            uint32_t c[8];   // codes of weights 128h + 32qq + 4u .. 4u + 3
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t ql = B.w[16 * h + 8 * (qq & 1) + u], qh = B.w[32 + 8 * h + u];
                const uint32_t lo = qq < 2 ? ql : ql >> 4;
                const uint32_t hi = qq == 0 ? qh << 4 : qq == 1 ? qh << 2 : qq == 2 ? qh : qh >> 2;
                c[u] = (lo & 0x0F0F0F0Fu) | (hi & 0x30303030u);
            }
            const int g = 8 * h + 2 * qq;   // groups g (u < 4) and g + 1
            const uint32_t sw = B.w[48 + (g >> 2)];
            const int s0 = (int)(int8_t)(uint8_t)(sw >> (8 * (g & 3)));
            const int s1 = (int)(int8_t)(uint8_t)(sw >> (8 * (g & 3) + 8));
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const uint8_t* a = act + (size_t)i * act_stride;
                const int4 x0 = *reinterpret_cast<const int4*>(a + 128 * h + 32 * qq);
                const int4 x1 = *reinterpret_cast<const int4*>(a + 128 * h + 32 * qq + 16);
                const int bs = *reinterpret_cast<const int*>(a + 256 + 2 * g);   // bsums g, g + 1
                int d0 = dp4a_us(c[0], x0.x, 0);
                d0 = dp4a_us(c[1], x0.y, d0);
                d0 = dp4a_us(c[2], x0.z, d0);
                d0 = dp4a_us(c[3], x0.w, d0);
                int d1 = dp4a_us(c[4], x1.x, 0);
                d1 = dp4a_us(c[5], x1.y, d1);
                d1 = dp4a_us(c[6], x1.z, d1);
                d1 = dp4a_us(c[7], x1.w, d1);
                d0 -= 32 * (int)(int16_t)(bs & 0xFFFF);
                d1 -= 32 * (bs >> 16);
                if constexpr (SUBDOTS) {
                    sub[i * sub_stride + g] = d0;
                    sub[i * sub_stride + g + 1] = d1;
                } else {
                    isum[i] += s0 * d0 + s1 * d1;
                }
            }
        }
    }
    if constexpr (!SUBDOTS) {
        const float d = half_bits_to_float(B.d);
#pragma unroll
        for (int i = 0; i < M; ++i) v[i] = __fmaf_rn(dy[i * dy_stride], __fmul_rn(d, (float)isum[i]), v[i]);
    }
}

// One whole q2_K or q3_K block against M staged activation blocks (records
// as for q6_K).  Weight 128h + 32j + 16p + l takes its two low bits from
// bits 2j, 2j + 1 of qs[32h + 16p + l]; q3_K adds bit 4h + j of
// hmask[16p + l] as the third bit (code q3 + 4 in 0..7, corrected by
// 4 bsum).  q2_K: isum = sum of sc * dot, msum = sum of m * bsum over the
// sixteen groups, term d (d isum - dmin msum) as for q4_K; q3_K: scale
// s - 32 from its six bits (low four from scales[g % 8], nibble g / 8, top
// two from scales[8 + g % 4], bits 2 (g / 4)), isum = sum of s * dot -
// 4 sum of s * bsum.  The sixteen exact group dots go to the export (q2_K
// the raw code dots, q3_K the corrected ones, as the four-lane kernel
// writes them).
//
// Without the export (every m of q2_K, m <= 3 of q3_K: above, the form's
// extra registers spill) the codes stay where they sit in the qs word: plane j
// is masked, not shifted, so each byte holds 4^e times its code (e = j; for
// q3_K e = min(j, 2), since the third bit must fit in the byte), and the dot
// comes out 4^e times too large.  The group pair's sum s0 dot0 + s1 dot1 is
// then multiplied by 4^(3 - e) instead, every plane ends up 64 times too
// large, and the sum is divided by 64 once per block (exactly: it is a
// multiple of 64).  The min term (q2_K) and the 4 bsum correction (q3_K) are
// one two-way dot of the pair's bsums with its two mins or scales.
template <int FMT, int M, bool SUBDOTS>
__device__ __forceinline__ void lane_block_q23(const WordBlock<FMT>& B, const uint8_t* act, int act_stride,
                                               const float* dy, int dy_stride, float* v, int32_t* sub,
                                               size_t sub_stride) {
    // the in-place form for every m of q2_K and for m <= 3 of q3_K (above, its extra
    // registers spill); the export and the other q3_K cases take the codes shifted down
    constexpr bool INPLACE = !SUBDOTS && (FMT == 2 || M <= 3);
    if constexpr (!INPLACE) {
        constexpr int QSW = LaneFmt<FMT>::QS / 4;   // first qs word
        int isum[M], msum[M];
#pragma unroll
        for (int i = 0; i < M; ++i) isum[i] = msum[i] = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t c[8];   // codes of weights 128h + 32j + 4u .. 4u + 3
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    c[u] = (B.w[QSW + 8 * h + u] >> (2 * j)) & 0x03030303u;
                    if constexpr (FMT == 3) c[u] |= ((B.w[u] >> (4 * h + j)) & 0x01010101u) << 2;
                }
                const int g = 8 * h + 2 * j;   // groups g (u < 4) and g + 1
                int s0, s1, m0 = 0, m1 = 0;
                if constexpr (FMT == 2) {
                    const uint32_t sb = B.w[g >> 2] >> (8 * (g & 3));   // scale bytes g, g + 1
                    s0 = (int)(sb & 15u);
                    m0 = (int)((sb >> 4) & 15u);
                    s1 = (int)((sb >> 8) & 15u);
                    m1 = (int)((sb >> 12) & 15u);
                } else {
                    auto scale = [&](int gg) {
                        const int lb = gg & 7, hb = 8 + (gg & 3);
                        const uint32_t low = (B.w[24 + (lb >> 2)] >> (8 * (lb & 3) + 4 * (gg >> 3))) & 15u;
                        const uint32_t high = (B.w[24 + (hb >> 2)] >> (8 * (hb & 3) + 2 * (gg >> 2))) & 3u;
                        return (int)(low | (high << 4)) - 32;
                    };
                    s0 = scale(g);
                    s1 = scale(g + 1);
                }
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    const uint8_t* a = act + (size_t)i * act_stride;
                    const int4 x0 = *reinterpret_cast<const int4*>(a + 128 * h + 32 * j);
                    const int4 x1 = *reinterpret_cast<const int4*>(a + 128 * h + 32 * j + 16);
                    const int bs = *reinterpret_cast<const int*>(a + 256 + 2 * g);   // bsums g, g + 1
                    const int b0 = (int)(int16_t)(bs & 0xFFFF), b1 = bs >> 16;
                    int d0 = dp4a_us(c[0], x0.x, 0);
                    d0 = dp4a_us(c[1], x0.y, d0);
                    d0 = dp4a_us(c[2], x0.z, d0);
                    d0 = dp4a_us(c[3], x0.w, d0);
                    int d1 = dp4a_us(c[4], x1.x, 0);
                    d1 = dp4a_us(c[5], x1.y, d1);
                    d1 = dp4a_us(c[6], x1.z, d1);
                    d1 = dp4a_us(c[7], x1.w, d1);
                    if constexpr (FMT == 3) {
                        d0 -= 4 * b0;
                        d1 -= 4 * b1;
                    }
                    if constexpr (SUBDOTS) {
                        sub[i * sub_stride + g] = d0;
                        sub[i * sub_stride + g + 1] = d1;
                    } else {
                        isum[i] += s0 * d0 + s1 * d1;
                        if constexpr (FMT == 2) msum[i] += m0 * b0 + m1 * b1;
                    }
                }
            }
        }
        if constexpr (!SUBDOTS) {
            if constexpr (FMT == 2) {
                const float d = half_bits_to_float(B.w[20]), dmin = half_bits_to_float(B.w[20] >> 16);
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    const float tt = __fmaf_rn(d, (float)isum[i], -__fmul_rn(dmin, (float)msum[i]));
                    v[i] = __fmaf_rn(dy[i * dy_stride], tt, v[i]);
                }
            } else {
                const float d = half_bits_to_float(B.d);
#pragma unroll
                for (int i = 0; i < M; ++i) v[i] = __fmaf_rn(dy[i * dy_stride], __fmul_rn(d, (float)isum[i]), v[i]);
            }
        }
    } else {
        constexpr int QSW = LaneFmt<FMT>::QS / 4;   // first qs word
        auto scale3 = [&](int gg) {   // q3_K: the signed 6-bit scale of group gg
            const int lb = gg & 7, hb = 8 + (gg & 3);
            const uint32_t low = (B.w[24 + (lb >> 2)] >> (8 * (lb & 3) + 4 * (gg >> 3))) & 15u;
            const uint32_t high = (B.w[24 + (hb >> 2)] >> (8 * (hb & 3) + 2 * (gg >> 2))) & 3u;
            return (int)(low | (high << 4)) - 32;
        };
        int iacc[M], bacc[M];   // 64 sum_g s_g dot_g; q2_K sum_g m_g bsum_g, q3_K sum_g s_g bsum_g
#pragma unroll
        for (int i = 0; i < M; ++i) iacc[i] = bacc[i] = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = FMT == 3 && j == 3 ? 2 : j;   // the plane's bytes hold 4^e x the code
                uint32_t c[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t w = B.w[QSW + 8 * h + u];
                    c[u] = (e == j ? w : w >> 2) & (0x03030303u << (2 * e));
                    if constexpr (FMT == 3) {   // the third bit, from bit 4h + j to bit 2e + 2
                        const uint32_t hb = B.w[u] & (0x01010101u << (4 * h + j));
                        const int sh = 2 * e + 2 - (4 * h + j);
                        c[u] |= sh >= 0 ? hb << sh : hb >> -sh;
                    }
                }
                const int g = 8 * h + 2 * j;   // groups g (u < 4) and g + 1
                int s0, s1;
                uint32_t pair;   // bytes 0, 1: q2_K the two mins, q3_K the two scales (signed)
                if constexpr (FMT == 2) {
                    const uint32_t sb = B.w[g >> 2] >> (8 * (g & 3));   // scale bytes g, g + 1
                    s0 = (int)(sb & 15u);
                    s1 = (int)((sb >> 8) & 15u);
                    pair = (sb >> 4) & 0x0F0Fu;
                } else {
                    s0 = scale3(g);
                    s1 = scale3(g + 1);
                    pair = __byte_perm((uint32_t)s0, (uint32_t)s1, 0x0040u);
                }
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    const uint8_t* a = act + (size_t)i * act_stride;
                    const int4 x0 = *reinterpret_cast<const int4*>(a + 128 * h + 32 * j);
                    const int4 x1 = *reinterpret_cast<const int4*>(a + 128 * h + 32 * j + 16);
                    const int bs = *reinterpret_cast<const int*>(a + 256 + 2 * g);   // bsums g, g + 1
                    int d0 = dp4a_us(c[0], x0.x, 0);
                    d0 = dp4a_us(c[1], x0.y, d0);
                    d0 = dp4a_us(c[2], x0.z, d0);
                    d0 = dp4a_us(c[3], x0.w, d0);
                    int d1 = dp4a_us(c[4], x1.x, 0);
                    d1 = dp4a_us(c[5], x1.y, d1);
                    d1 = dp4a_us(c[6], x1.z, d1);
                    d1 = dp4a_us(c[7], x1.w, d1);
                    iacc[i] += (s0 * d0 + s1 * d1) * (1 << (6 - 2 * e));
                    if constexpr (FMT == 2)
                        bacc[i] = dp2a_lo_su(bs, pair, bacc[i]);
                    else
                        bacc[i] = dp2a_lo_ss(bs, pair, bacc[i]);
                }
            }
        }
        if constexpr (FMT == 2) {
            const float d = half_bits_to_float(B.w[20]), dmin = half_bits_to_float(B.w[20] >> 16);
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const float tt = __fmaf_rn(d, (float)(iacc[i] >> 6), -__fmul_rn(dmin, (float)bacc[i]));
                v[i] = __fmaf_rn(dy[i * dy_stride], tt, v[i]);
            }
        } else {
            const float d = half_bits_to_float(B.d);
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const int isum = (iacc[i] >> 6) - 4 * bacc[i];
                v[i] = __fmaf_rn(dy[i * dy_stride], __fmul_rn(d, (float)isum), v[i]);
            }
        }
    }
}

template <int FMT, int M, bool SUBDOTS, bool XF32, bool PAIR, int WARPS, int MAXP>
__global__ void __launch_bounds__(WARPS * 32, 1) lane_kernel(const __grid_constant__ LaneBatch<MAXP> B) {
    constexpr int PF = PAIR ? 2 : 1;
    constexpr int BYTES = LaneFmt<FMT>::BYTES;
    constexpr int SLOT = slot_bytes<FMT>();
    constexpr int REC = rec_bytes<FMT>();
    constexpr int SUBN = sub_per_block<FMT>();
    static_assert(!XF32 || FMT == 4, "the fused producer stages q4_K records");
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int NS = B.nstages;
    uint8_t* ring = smem + B.act_bytes + (size_t)warp * NS * SLOT;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + B.act_bytes + (size_t)WARPS * NS * SLOT) + warp * NS;
    if (lane == 0) {
        for (int j = 0; j < NS; ++j) mbar_init(&bars[j], 1);
        fence_barrier_init();
    }
    __syncwarp();
    grid_launch_dependents();

    // even split of the weighted units over all warps of the grid
    const long long G = (long long)gridDim.x * WARPS;
    const long long gw = (long long)blockIdx.x * WARPS + warp;
    const int W0 = (int)(B.wtotal * gw / G), W1 = (int)(B.wtotal * (gw + 1) / G);
    const int C0 = (int)(B.wtotal * ((long long)blockIdx.x * WARPS) / G);
    const int C1 = (int)(B.wtotal * ((long long)blockIdx.x * WARPS + WARPS) / G);

    // copy cursor: lane 0 issues; runs up to NS stages ahead, across problems
    Cursor ic;
    cursor_enter(B, ic, problem_at(B, W0), W0, W1, PF);
    uint32_t issued = 0, consumed = 0;           // ring counters, uniform in the warp
    uint32_t islot = 0, cslot = 0, cphase = 0;   // next slot to fill / to consume, its phase parity
    auto issue_one = [&]() {
        const LaneProblem& Q = B.p[ic.p];
        const int nb = Q.nb;
        const int spr = unit_weight(nb);
        const bool second = PAIR && ic.ch >= spr;   // paired: the up matrix's stages follow the gate's
        const int ch = second ? ic.ch - spr : ic.ch;
        int blocks;
        long long first;   // first block of the stage
        if (nb <= STAGE_BLOCKS) {
            const int r0 = ic.u * Q.rps;
            blocks = min(Q.rps, Q.n - r0) * nb;
            first = (long long)r0 * nb;
        } else {
            const int b0 = ch * STAGE_BLOCKS;
            blocks = min(STAGE_BLOCKS, nb - b0);
            first = (long long)ic.u * nb + b0;
        }
        if (lane == 0) {
            uint64_t* bar = &bars[islot];
            const uint32_t bytes = (uint32_t)blocks * BYTES;   // rows: whole 16-byte multiples
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(ring + islot * SLOT, (second ? Q.w2 : Q.w) + first * BYTES, bytes, bar);
        }
        islot = islot + 1 == (uint32_t)NS ? 0 : islot + 1;
        ++issued;
        cursor_next(B, ic, nb, W0, W1, PF);
    };
    // stage the activations of every problem the CTA's warps touch, filling
    // the ring once the first activation loads are out
    const int cfirst = problem_at(B, C0);
    int cend = cfirst;
    while (cend < B.count && B.p[cend].wbegin < C1) ++cend;
    auto fill = [&]() {
        while (ic.p >= 0 && issued < (uint32_t)NS) issue_one();
    };
    // weights first when they may be copied before the earlier kernels end
    // (nothing before this launch writes them); activations only after
    if (B.prefetch) fill();
    grid_wait_prior();
    if constexpr (XF32)
        stage_f32<M, WARPS>(B, cfirst, cend, smem, warp, lane, fill);
    else
        stage_q8<FMT, M, 8>(B, cfirst, cend, smem, fill);
    __syncthreads();

    Cursor cc;
    cursor_enter(B, cc, problem_at(B, W0), W0, W1, PF);
    int act_p = cfirst, act_off = 0;   // staged offset of problem act_p
    bool ok = true;                    // false once a wait ran out
    while (cc.p >= 0 && ok) {
        // per problem: geometry and pointers
        const LaneProblem& P = B.p[cc.p];
        const int p_now = cc.p;
        const int nb = P.nb, n = P.n, rps = P.rps;
        while (act_p < p_now) {
            act_off += seg_bytes<FMT>(M * B.p[act_p].nb);
            ++act_p;
        }
        const uint8_t* rec = smem + act_off;
        const float* dyv = reinterpret_cast<const float*>(rec + (size_t)M * nb * REC);
        const int act_stride = nb * REC;
        const size_t sub_stride = (size_t)n * nb * SUBN;
        float* yv = P.y;
        int32_t* subv = P.sub;
        const int rl = rps > 0 ? lane / nb : 0;   // row mode: row slot and column of this lane
        const int cl = rps > 0 ? lane - rl * nb : lane;
        const bool pow2 = (nb & (nb - 1)) == 0;
        float acc[M], gsum[M];   // gsum: paired launches, the gate row sums
#pragma unroll
        for (int i = 0; i < M; ++i) acc[i] = gsum[i] = 0.0f;

        while (cc.p == p_now) {
            if (!mbar_wait(&bars[cslot], cphase)) {
                // a copy never completed: record it, let our other copies land, stop
                if (lane == 0) {
                    atomicOr(B.fault, 1u);
                    for (uint32_t c2 = consumed; c2 < issued; ++c2) (void)mbar_wait(&bars[c2 % NS], (c2 / NS) & 1);
                }
                __syncwarp();
                ok = false;
                break;
            }
            const uint8_t* slot = ring + cslot * SLOT;
            // this lane's block of the stage (clamped to block 0 when it has none; result discarded)
            const int lane_blk = rps > 0 ? (rl < min(rps, n - cc.u * rps) ? lane : 0)
                                         : (lane < min(STAGE_BLOCKS, nb - stage_b0(cc.ch, nb)) ? lane : 0);
            // m <= 2: copy the block into registers and refill the slot at once,
            // so every stage of the ring is in flight while this one is decoded
            constexpr bool EARLY = !SUBDOTS && M <= 2;
            constexpr bool WORDS = FMT == 2 || FMT == 3 || FMT == 6;   // blocks read as 4-byte words
            typename std::conditional<WORDS, WordBlock<WORDS ? FMT : 6>, RegBlock<BYTES / 16>>::type rb;
            if constexpr (EARLY) {
                if constexpr (WORDS) {
                    word_block_load<FMT>(slot + lane_blk * BYTES, rb);
                } else {
#pragma unroll
                    for (int u = 0; u < BYTES / 16; ++u)
                        rb.r[u] = reinterpret_cast<const uint4*>(slot + lane_blk * BYTES)[u];
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // reads before the refill
                ++consumed;
                if (++cslot == (uint32_t)NS) {
                    cslot = 0;
                    cphase ^= 1u;
                }
                __syncwarp();
                if (ic.p >= 0) issue_one();
            }
            auto decode = [&](const uint8_t* act, const float* dyp, float* v, int32_t* sub) {
                if constexpr (WORDS) {
                    WordBlock<WORDS ? FMT : 6> wb;
                    if constexpr (EARLY)
                        wb = rb;
                    else
                        word_block_load<FMT>(slot + lane_blk * BYTES, wb);
                    if constexpr (FMT == 6)
                        lane_block_q6<M, SUBDOTS>(wb, act, act_stride, dyp, nb, v, sub, sub_stride);
                    else
                        lane_block_q23<FMT, M, SUBDOTS>(wb, act, act_stride, dyp, nb, v, sub, sub_stride);
                } else if constexpr (EARLY) {
                    lane_block<FMT, M, SUBDOTS>(rb, act, act_stride, dyp, nb, v, sub, sub_stride);
                } else {
                    lane_block<FMT, M, SUBDOTS>(SmemBlock{slot + lane_blk * BYTES}, act, act_stride, dyp, nb, v, sub,
                                                sub_stride);
                }
            };
            if (rps > 0) {
                const int r0 = cc.u * rps;
                const int nrows = min(rps, n - r0);
                const bool valid = rl < nrows;
                const int col = valid ? cl : 0;
                float v[M];
#pragma unroll
                for (int i = 0; i < M; ++i) v[i] = 0.0f;
                int32_t* sub = SUBDOTS ? subv + ((size_t)(r0 + rl) * nb + col) * SUBN : nullptr;
                if (!SUBDOTS || valid) decode(rec + (size_t)col * REC, dyv + col, v, sub);
                if constexpr (!SUBDOTS) {
                    if (pow2) {
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1)
                            if (o < nb) {
#pragma unroll
                                for (int i = 0; i < M; ++i) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], o);
                            }
                    } else {
#pragma unroll
                        for (int o = 1; o <= 16; o <<= 1) {
#pragma unroll
                            for (int i = 0; i < M; ++i) {
                                const float u = __shfl_down_sync(0xFFFFFFFFu, v[i], o);
                                if (cl + o < nb) v[i] += u;
                            }
                        }
                    }
                    if (PAIR && cc.ch == 0) {
#pragma unroll
                        for (int i = 0; i < M; ++i) gsum[i] = v[i];
                    } else if (valid && cl == 0) {
#pragma unroll
                        for (int i = 0; i < M; ++i) yv[(size_t)i * n + r0 + rl] = PAIR ? swiglu(gsum[i], v[i]) : v[i];
                    }
                }
            } else {
                const int spr = unit_weight(nb);
                const bool second = PAIR && cc.ch >= spr;
                const int b0 = (second ? cc.ch - spr : cc.ch) * STAGE_BLOCKS;
                const int nblk_s = min(STAGE_BLOCKS, nb - b0);
                const bool valid = lane < nblk_s;
                const int b = b0 + (valid ? lane : 0);
                float v[M];
#pragma unroll
                for (int i = 0; i < M; ++i) v[i] = acc[i];
                int32_t* sub = SUBDOTS ? subv + ((size_t)cc.u * nb + b) * SUBN : nullptr;
                if (!SUBDOTS || valid) decode(rec + (size_t)b * REC, dyv + b, v, sub);
#pragma unroll
                for (int i = 0; i < M; ++i) acc[i] = valid ? v[i] : acc[i];
                if (b0 + STAGE_BLOCKS >= nb) {   // last stage of the row
                    if constexpr (!SUBDOTS) {
#pragma unroll
                        for (int i = 0; i < M; ++i) {
                            const float x = warp_sum(acc[i]);
                            if (PAIR && !second)
                                gsum[i] = x;
                            else if (lane == 0)
                                yv[(size_t)i * n + cc.u] = PAIR ? swiglu(gsum[i], x) : x;
                            acc[i] = 0.0f;
                        }
                    }
                }
            }
            if constexpr (!EARLY) {
                ++consumed;
                if (++cslot == (uint32_t)NS) {
                    cslot = 0;
                    cphase ^= 1u;
                }
                __syncwarp();
                if (ic.p >= 0) issue_one();
            }
            cursor_next(B, cc, nb, W0, W1, PF);
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct Config {
    int warps, ns, grid, act_bytes;
};


template <int FMT>
inline size_t ring_bytes(int warps, int ns) { return (size_t)warps * ns * (slot_bytes<FMT>() + 8); }
inline size_t align128(size_t x) { return (x + 127) & ~(size_t)127; }

struct Plan {
    int rps[GROUP_MAX], wbegin[GROUP_MAX];
    long long wtotal;
};

// Units per problem.  A launch too small to give every warp of the GPU two
// units takes fewer rows per unit (down to one), so that its rows still
// spread over all SMs; rows per unit do not change any row's arithmetic.
inline void make_plan(const HostProblem* hp, int count, int warps, int pairf, Plan* pl) {
    const long long target = 2LL * num_sms() * warps;
    for (int shrink = 1;; shrink *= 2) {
        long long w = 0;
        bool reducible = false;
        for (int i = 0; i < count; ++i) {
            const int nb = hp[i].nb;
            const int full = nb <= STAGE_BLOCKS ? STAGE_BLOCKS / nb : 0;
            pl->rps[i] = full > 0 ? std::max(1, full / shrink) : 0;
            reducible = reducible || pl->rps[i] > 1;
            pl->wbegin[i] = (int)std::min(w, (long long)INT32_MAX);
            w += (long long)unit_count(hp[i].n, pl->rps[i]) * unit_stages(nb, pairf);
        }
        pl->wtotal = w;
        if (w >= target || !reducible) return;
    }
}

// Largest staged-activation region over the CTAs: every problem whose
// weighted range meets the CTA's (the kernel stages the same set).
template <int FMT>
inline size_t act_need(const HostProblem* hp, int count, const Plan& pl, int m, int grid, int warps) {
    const long long G = (long long)grid * warps;
    size_t worst = 0;
    int p = 0;
    for (int c = 0; c < grid; ++c) {
        const long long C0 = pl.wtotal * ((long long)c * warps) / G;
        const long long C1 = pl.wtotal * ((long long)c * warps + warps) / G;
        while (p + 1 < count && pl.wbegin[p + 1] <= C0) ++p;
        size_t sum = 0;
        for (int q = p; q < count && pl.wbegin[q] < C1; ++q) sum += (size_t)seg_bytes<FMT>(m * hp[q].nb);
        worst = std::max(worst, sum);
    }
    return align128(worst);
}

template <int FMT>
inline bool pick_config(const HostProblem* hp, int count, const Plan& pl, int m, Config* cfg) {
    const size_t optin = (size_t)smem_optin_bytes();
    const int opts[][2] = {{16, 3}, {16, 2}, {12, 2}};
    for (const auto& o : opts) {
        long long grid = num_sms();
        const long long want = (pl.wtotal + o[0] - 1) / o[0];   // no CTA without a unit per warp
        if (grid > want) grid = want;
        if (grid < 1) grid = 1;
        const size_t act = act_need<FMT>(hp, count, pl, m, (int)grid, o[0]);
        if (act + ring_bytes<FMT>(o[0], o[1]) <= optin) {
            *cfg = Config{o[0], o[1], (int)grid, (int)act};
            return true;
        }
    }
    return false;
}

template <int FMT, int M, bool SUB, bool XF32, bool PAIR, int WARPS, int MAXP>
cudaError_t launch(const HostProblem* hp, int count, const Plan& pl, const Config& cfg, cudaStream_t stream) {
    LaneBatch<MAXP> B;
    B.fault = fault_word();
    if (!B.fault) return cudaErrorInvalidDevicePointer;
    for (int i = 0; i < count; ++i) {
        B.p[i] = LaneProblem{hp[i].w,  hp[i].xq, hp[i].y,      hp[i].sub, hp[i].n,
                             hp[i].nb, pl.rps[i], pl.wbegin[i], hp[i].w2};
    }
    B.count = count;
    B.nstages = cfg.ns;
    B.act_bytes = cfg.act_bytes;
    B.wtotal = (int)pl.wtotal;
    B.prefetch = overlap_mode() >= 2 ? 1 : 0;
    const size_t smem = (size_t)cfg.act_bytes + ring_bytes<FMT>(WARPS, cfg.ns);
    const void* fn = (const void*)lane_kernel<FMT, M, SUB, XF32, PAIR, WARPS, MAXP>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(lane_kernel<FMT, M, SUB, XF32, PAIR, WARPS, MAXP>, dim3((unsigned)cfg.grid),
                         dim3(WARPS * 32), smem, stream, B);
}

// Launches one pass of M activation rows; false in *fits when no ring and
// staging layout fits in shared memory (the caller then splits the work).
template <int FMT, int M, bool SUB, bool XF32, bool PAIR>
cudaError_t launch_m(const HostProblem* hp, int count, cudaStream_t stream, bool* fits) {
    Plan pl;
    make_plan(hp, count, 16, PAIR ? 2 : 1, &pl);
    *fits = false;
    if (pl.wtotal >= (1LL << 31)) return cudaSuccess;
    Config cfg;
    if (!pick_config<FMT>(hp, count, pl, M, &cfg)) return cudaSuccess;
    *fits = true;
    if (cfg.warps == 16) {
        if (count == 1) return launch<FMT, M, SUB, XF32, PAIR, 16, 1>(hp, count, pl, cfg, stream);
        if constexpr (!SUB) return launch<FMT, M, SUB, XF32, PAIR, 16, GROUP_MAX>(hp, count, pl, cfg, stream);
    } else {
        if (count == 1) return launch<FMT, M, SUB, XF32, PAIR, 12, 1>(hp, count, pl, cfg, stream);
        if constexpr (!SUB) return launch<FMT, M, SUB, XF32, PAIR, 12, GROUP_MAX>(hp, count, pl, cfg, stream);
    }
    return cudaErrorInvalidValue;
}

template <int FMT, bool SUB, bool XF32, bool PAIR>
cudaError_t dispatch(int m, const HostProblem* hp, int count, cudaStream_t stream, bool* fits) {
    switch (m) {
        case 1: return launch_m<FMT, 1, SUB, XF32, PAIR>(hp, count, stream, fits);
        case 2: return launch_m<FMT, 2, SUB, XF32, PAIR>(hp, count, stream, fits);
        case 3: return launch_m<FMT, 3, SUB, XF32, PAIR>(hp, count, stream, fits);
        case 4: return launch_m<FMT, 4, SUB, XF32, PAIR>(hp, count, stream, fits);
        case 5: return launch_m<FMT, 5, SUB, XF32, PAIR>(hp, count, stream, fits);
        case 6: return launch_m<FMT, 6, SUB, XF32, PAIR>(hp, count, stream, fits);
        case 7: return launch_m<FMT, 7, SUB, XF32, PAIR>(hp, count, stream, fits);
        case 8: return launch_m<FMT, 8, SUB, XF32, PAIR>(hp, count, stream, fits);
        default: return cudaErrorInvalidValue;
    }
}

// Runs problems [0, count) with activation rows [i0, i0 + mm): as one launch
// when it fits, else the problems in two halves; a single problem that does
// not fit is taken in smaller row passes.  The f32 order of an output row
// depends only on nb, so none of these splits changes a bit.
template <int FMT, bool XF32, bool PAIR>
cudaError_t run_part(const HostProblem* probs, int count, int i0, int mm, bool subdots, cudaStream_t stream) {
    HostProblem part[GROUP_MAX];
    for (int j = 0; j < count; ++j) {
        const HostProblem& s = probs[j];
        part[j] = s;
        // activation row i0: q8_K blocks, or f32 values when XF32
        part[j].xq = s.xq + (size_t)i0 * s.nb * (XF32 ? QK * sizeof(float) : Q8K_BYTES);
        part[j].y = s.y ? s.y + (size_t)i0 * s.n : nullptr;
        part[j].sub = s.sub ? s.sub + (size_t)i0 * s.n * s.nb * sub_per_block<FMT>() : nullptr;
    }
    bool fits = false;
    cudaError_t e;
    if constexpr (XF32 || PAIR)
        e = dispatch<FMT, false, XF32, PAIR>(mm, part, count, stream, &fits);
    else
        e = subdots ? dispatch<FMT, true, false, false>(mm, part, count, stream, &fits)
                    : dispatch<FMT, false, false, false>(mm, part, count, stream, &fits);
    if (e != cudaSuccess || fits) return e;
    if (count > 1) {
        const int h = count / 2;
        e = run_part<FMT, XF32, PAIR>(probs, h, i0, mm, subdots, stream);
        if (e != cudaSuccess) return e;
        return run_part<FMT, XF32, PAIR>(probs + h, count - h, i0, mm, subdots, stream);
    }
    if (mm == 1) return cudaErrorInvalidConfiguration;
    const int h = mm / 2;
    e = run_part<FMT, XF32, PAIR>(probs, 1, i0, h, subdots, stream);
    if (e != cudaSuccess) return e;
    return run_part<FMT, XF32, PAIR>(probs, 1, i0 + h, mm - h, subdots, stream);
}

template <int FMT, bool XF32, bool PAIR>
cudaError_t run_group(const HostProblem* probs, int count, int m, bool subdots, cudaStream_t stream) {
    for (int p0 = 0; p0 < count; p0 += GROUP_MAX) {
        const int cnt = count - p0 < GROUP_MAX ? count - p0 : GROUP_MAX;
        const cudaError_t e = run_part<FMT, XF32, PAIR>(probs + p0, cnt, 0, m, subdots, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// q2_K, q3_K, q6_K: this kernel takes a problem whose rows hold a multiple
// of four (q2_K) or eight blocks (so every stage copy starts and ends on a
// 16-byte boundary), whose matrix starts on a 16-byte boundary and one of
// whose activation rows fits beside the smallest ring; the four-lanes-per-
// block kernel of gemv_impl.cuh takes the others.  The choice depends on
// the problem alone (not on m or on the rest of its group), so a row's bits
// are the same for every m and every grouping.
template <int FMT>
inline bool lane_eligible(const HostProblem& p) {
    constexpr int ROWS_OF = FMT == 2 ? 4 : 8;
    return p.nb % ROWS_OF == 0 && ((uintptr_t)p.w & 15u) == 0 &&
           align128((size_t)seg_bytes<FMT>(p.nb)) + ring_bytes<FMT>(12, 2) <= (size_t)smem_optin_bytes();
}

template <int FMT>
cudaError_t run_group_words(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream) {
    if (count > GROUP_MAX) return cudaErrorInvalidValue;   // callers pass at most GROUP_MAX problems
    HostProblem lane[GROUP_MAX], quad[GROUP_MAX];
    int nl = 0, nq = 0;
    for (int i = 0; i < count; ++i) {
        if (lane_eligible<FMT>(p[i]))
            lane[nl++] = p[i];
        else
            quad[nq++] = p[i];
    }
    cudaError_t e = cudaSuccess;
    if (nl > 0) e = run_group<FMT, false, false>(lane, nl, m, subdots, stream);
    if (e == cudaSuccess && nq > 0) e = plm::run_group<FMT>(quad, nq, m, subdots, stream);
    return e;
}

}  // namespace q4lane
}  // namespace plm
