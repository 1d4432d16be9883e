// Decode GEMV for m = 1..8 activation rows over packed q6_K weights (the
// output head) and the low rungs q2_K and q3_K (PocketLLM "What it runs":
// K-quant weights decoded inside the kernel, never widened; the weight stream
// is read once for all m activation rows, as the pages' 8-row activation tile
// does on the CPU), for the problems the one-lane-per-block kernel of
// gemv_q4K.cuh does not take: rows whose blocks would leave a stage copy off
// a 16-byte boundary (q6_K, q3_K: a multiple of eight blocks; q2_K: four).
// q4_K and q5_K always take that kernel; the host problem descriptor here is
// shared with it.
//
// One launch serves a group of independent problems {w, xq, y, n, k} that
// share m (a single GEMV is a group of one).  The weight bytes of all
// problems form one flat byte space, split evenly across persistent CTAs
// (one per SM, 16 warps each).  A CTA walks the problem segments that fall in its
// range; for each it stages the problem's q8_K activations in shared memory
// and splits the segment's rows across its warps.
//
// Each warp streams its rows (one contiguous byte range of W) through its
// own ring of shared-memory stages filled by 1-D bulk copies
// (cp.async.bulk, completion counted on one mbarrier per stage).  A stage
// holds whole rows when a row is small, else a 16-block chunk of one row.
// The first copies of a segment are issued before the CTA stages that
// segment's activations, so the two overlap.  Every wait is bounded; a wait
// that runs out records a fault and the warp stops computing (it still
// takes part in every CTA barrier).
//
// Four lanes share one 256-weight block, so a warp handles eight blocks per
// step; a lane owns four whole 16-weight groups.  Per block and activation
// row a lane forms exact integer dots with dp4a, applies the group scales in
// int32 and adds one f32 term.  When nb divides 8, one step covers 8/nb
// whole rows and each row is reduced over its own 4*nb lanes; otherwise a
// row takes ceil(nb/8) steps and is reduced over the warp.  The f32 order
// of a row depends only on nb (explicit _rn intrinsics), so activation row
// i gives the same bits for every m and every grouping.
//
// q6_K blocks are 210 bytes, so blocks are only 2-byte aligned.  A stage's
// copy starts at the 16-byte boundary below its first block; fields are read
// back with aligned loads and funnel shifts.  The last bytes of the matrix,
// past its final 16-byte boundary, are read with plain loads.
//
// With SUBDOTS the same kernel writes the integer sub-block dots instead of
// the f32 result (verification export).
#pragma once

#include <type_traits>

#include "plm_device.cuh"
#include "plm_internal.h"

namespace plm {

constexpr int BLOCKS_PER_STEP = 8;     // 32 lanes, 4 per block
constexpr int MAX_STAGES = 8;
constexpr int GEMV_WARPS = 16;
constexpr int GROUP_MAX = 256;         // problems per grouped launch

template <int FMT> struct Fmt;
template <> struct Fmt<6> {
    static constexpr int BYTES = Q6K_BYTES;
    static constexpr int CHUNK = 16;
    static constexpr int PAYLOAD = CHUNK * Q6K_BYTES;          // 3360
    static constexpr int SLOT = 3456;                          // + 16-byte alignment slack
    static constexpr int SUB = 16;
};
template <> struct Fmt<2> {                                    // q2_K: 84-byte blocks, 4-byte aligned
    static constexpr int BYTES = Q2K_BYTES;
    static constexpr int CHUNK = 32;
    static constexpr int PAYLOAD = CHUNK * Q2K_BYTES;          // 2688
    static constexpr int SLOT = 2720;
    static constexpr int SUB = 16;
};
template <> struct Fmt<3> {                                    // q3_K: 110-byte blocks, 2-byte aligned
    static constexpr int BYTES = Q3K_BYTES;
    static constexpr int CHUNK = 32;
    static constexpr int PAYLOAD = CHUNK * Q3K_BYTES;          // 3520
    static constexpr int SLOT = 3552;
    static constexpr int SUB = 16;
};

struct GemvProblem {
    const uint8_t* w;
    const uint8_t* xq;
    float* y;
    int32_t* sub;
    long long byte_begin;   // offset of this problem's W in the group's flat byte space
    int n, nb;
};

template <int MAXP>
struct GemvBatch {
    unsigned* fault;
    long long total_bytes;
    int count;
    int nstages;            // ring depth per warp
    int act_bytes;          // 128-aligned size of the staged-activation region
    int prefetch;           // copy weights before waiting for the kernels before this one
    GemvProblem p[MAXP];
};

__device__ __forceinline__ long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

// Geometry of one stage, from its first row and first block.
struct StageGeom {
    int nrows, nblk;        // rows covered; blocks per row (row-chunk mode: blocks of the chunk)
    int bytes, tail, delta; // bulk bytes, plain-load tail bytes, first block's offset in the slot
    long long src;          // 16-byte aligned source offset into W
};

template <int FMT>
__device__ __forceinline__ StageGeom stage_geom(int row, int b0, int wb, int rps, int nb, long long wbytes) {
    constexpr int BYTES = Fmt<FMT>::BYTES;
    StageGeom g;
    g.nrows = rps > 0 ? min(rps, wb - row) : 1;
    g.nblk = rps > 0 ? nb : min(Fmt<FMT>::CHUNK, nb - b0);
    const long long S = ((long long)row * nb + b0) * BYTES;
    const long long E = S + (long long)(rps > 0 ? g.nrows * nb : g.nblk) * BYTES;
    const long long A0 = S & ~15LL;
    long long end = (E + 15) & ~15LL;
    g.tail = 0;
    if (end > wbytes) {        // never read past the end of the matrix
        end = wbytes & ~15LL;
        g.tail = (int)(wbytes - end);
    }
    g.src = A0;
    g.bytes = (int)(end - A0);
    g.delta = (int)(S - A0);
    return g;
}

// The activation values one lane needs for one block of one activation row:
//   lane (h, p) (q2_K, q3_K, q6_K): chunks 8h+2qq+p for qq = 0..3, bsums 8h+2qq+p
// bw[0] packs the first two bsums (low half first), bw[1] the last two.
struct LaneAct {
    int4 x[4];
    int bw[2];
    float dy;
};

template <int FMT>
__device__ __forceinline__ LaneAct act_from_smem(const ActSmem& a, int blk, int t) {
    LaneAct r;
    r.dy = a.dy[blk];
    {
        const int h = t >> 1, p = t & 1;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) r.x[qq] = *act_chunk<6>(a, blk, 8 * h + 2 * qq + p);
        const int4 v = *reinterpret_cast<const int4*>(a.bs + (size_t)blk * 16 + 8 * h);
        // words hold groups (8h+2qq, 8h+2qq+1); keep the half with parity p
        const int g0 = p ? (v.x >> 16) : (v.x & 0xFFFF), g1 = p ? (v.y >> 16) : (v.y & 0xFFFF);
        const int g2 = p ? (v.z >> 16) : (v.z & 0xFFFF), g3 = p ? (v.w >> 16) : (v.w & 0xFFFF);
        r.bw[0] = (g0 & 0xFFFF) | (g1 << 16);
        r.bw[1] = (g2 & 0xFFFF) | (g3 << 16);
    }
    return r;
}

// Same values straight from the q8_K bytes in global memory (4-byte aligned
// blocks): used when a lane keeps its activations in registers.
template <int FMT>
__device__ __forceinline__ LaneAct act_from_global(const uint8_t* __restrict__ xq, int blk, int t) {
    LaneAct r;
    const uint8_t* base = xq + (size_t)blk * Q8K_BYTES;
    r.dy = __ldg(reinterpret_cast<const float*>(base));
    const uint32_t* qs = reinterpret_cast<const uint32_t*>(base + 4);
    const uint32_t* bsw = reinterpret_cast<const uint32_t*>(base + 260);
    {
        const int h = t >> 1, p = t & 1;
        int g[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const int c = 8 * h + 2 * qq + p;
            const uint32_t* cp = qs + 4 * c;
            r.x[qq] = make_int4((int)__ldg(cp), (int)__ldg(cp + 1), (int)__ldg(cp + 2), (int)__ldg(cp + 3));
            const uint32_t wv = __ldg(bsw + (c >> 1));
            g[qq] = p ? (int)(wv >> 16) : (int)(wv & 0xFFFF);
        }
        r.bw[0] = (g[0] & 0xFFFF) | (g[1] << 16);
        r.bw[1] = (g[2] & 0xFFFF) | (g[3] << 16);
    }
    return r;
}

__device__ __forceinline__ int lo16(int w) { return (int)(int16_t)(w & 0xFFFF); }
__device__ __forceinline__ int hi16(int w) { return w >> 16; }

// One q6_K block at an even offset of the slot: lane t = (h, p).
template <int M, bool SUBDOTS>
__device__ __forceinline__ void q6K_block(const uint8_t* slot, int off, const LaneAct* act, int b, int t,
                                          float* v, int32_t* sub_row, size_t sub_stride_i) {
    const int h = t >> 1, p = t & 1;
    const uint4 A = lds16_align2(slot, off + 64 * h + 16 * p);
    const uint4 Bq = lds16_align2(slot, off + 64 * h + 32 + 16 * p);
    const uint4 H = lds16_align2(slot, off + 128 + 32 * h + 16 * p);
    const uint2 S = lds8_align2(slot, off + 192 + 8 * h);
    const uint32_t dbits = *reinterpret_cast<const uint16_t*>(slot + off + 208);
    const Q6KLane L = q6K_lane_decode(A, Bq, H, S, dbits, p);
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const LaneAct& X = act[i];
        const int bsum[4] = {lo16(X.bw[0]), hi16(X.bw[0]), lo16(X.bw[1]), hi16(X.bw[1])};
        int isum = 0;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const int dot = q6K_lane_raw(L, qq, X.x[qq]) - 32 * bsum[qq];
            if constexpr (SUBDOTS)
                sub_row[i * sub_stride_i + (size_t)b * 16 + 8 * h + 2 * qq + p] = dot;
            else
                isum += L.sc[qq] * dot;
        }
        if constexpr (!SUBDOTS) v[i] = __fmaf_rn(__fmul_rn(L.d, X.dy), (float)isum, v[i]);
    }
}


// q2_K / q3_K: lane t = (h, p) owns groups 8h + 2j + p, j = 0..3 -- the
// groups whose activations act_from_* gives it -- whose 2-bit codes are bits
// 2j, 2j+1 of the 16 bytes qs[32h + 16p .. +16]; q3_K's third bits are bit
// 4h + j of hmask[16p .. +16].
template <int M, bool SUBDOTS>
__device__ __forceinline__ void q2K_block(const uint8_t* slot, int off, const LaneAct* act, int b, int t,
                                          float* v, int32_t* sub_row, size_t sub_stride_i) {
    const int h = t >> 1, p = t & 1;
    const uint4 Q = lds16_align2(slot, off + 16 + 32 * h + 16 * p);
    const uint2 S = lds8_align2(slot, off + 8 * h);   // scale bytes 8h .. 8h+7: group 8h+2j+p at 2j+p
    const float d = half_bits_to_float(*reinterpret_cast<const uint16_t*>(slot + off + 80));
    const float dmin = half_bits_to_float(*reinterpret_cast<const uint16_t*>(slot + off + 82));
    const uint32_t qw[4] = {Q.x, Q.y, Q.z, Q.w};
    int sc[4], mn[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int byte = 2 * j + p;
        const uint32_t v8 = ((byte < 4 ? S.x : S.y) >> (8 * (byte & 3))) & 0xFFu;
        sc[j] = (int)(v8 & 15u);
        mn[j] = (int)(v8 >> 4);
    }
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const LaneAct& X = act[i];
        const int bsum[4] = {lo16(X.bw[0]), hi16(X.bw[0]), lo16(X.bw[1]), hi16(X.bw[1])};
        const int xs[4][4] = {{X.x[0].x, X.x[0].y, X.x[0].z, X.x[0].w}, {X.x[1].x, X.x[1].y, X.x[1].z, X.x[1].w},
                              {X.x[2].x, X.x[2].y, X.x[2].z, X.x[2].w}, {X.x[3].x, X.x[3].y, X.x[3].z, X.x[3].w}};
        int isum = 0, msum = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int dot = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) dot = dp4a_us((qw[u] >> (2 * j)) & 0x03030303u, xs[j][u], dot);
            if constexpr (SUBDOTS)
                sub_row[i * sub_stride_i + (size_t)b * 16 + 8 * h + 2 * j + p] = dot;
            isum += sc[j] * dot;
            msum += mn[j] * bsum[j];
        }
        if constexpr (!SUBDOTS) {
            const float tt = __fmaf_rn(d, (float)isum, -__fmul_rn(dmin, (float)msum));
            v[i] = __fmaf_rn(X.dy, tt, v[i]);
        }
    }
}

template <int M, bool SUBDOTS>
__device__ __forceinline__ void q3K_block(const uint8_t* slot, int off, const LaneAct* act, int b, int t,
                                          float* v, int32_t* sub_row, size_t sub_stride_i) {
    const int h = t >> 1, p = t & 1;
    const uint4 Q = lds16_align2(slot, off + 32 + 32 * h + 16 * p);
    const uint4 Hm = lds16_align2(slot, off + 16 * p);
    const uint4 T = lds16_align2(slot, off + 96);      // scales[12], then d
    const float d = half_bits_to_float(T.w);           // bytes 108, 109
    const uint32_t qw[4] = {Q.x, Q.y, Q.z, Q.w};
    const uint32_t hw[4] = {Hm.x, Hm.y, Hm.z, Hm.w};
    const uint32_t tw[3] = {T.x, T.y, T.z};
    int sc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // group g = 8h + 2j + p: low four bits from scales[2j + p] (nibble h),
        // top two from scales[8 + (2j + p) % 4], bits 2(2h + j/2)
        const int lb = 2 * j + p, hb = 8 + ((2 * j + p) & 3), hs = 2 * (2 * h + j / 2);
        const uint32_t low = ((tw[lb >> 2] >> (8 * (lb & 3) + 4 * h)) & 15u);
        const uint32_t high = ((tw[hb >> 2] >> (8 * (hb & 3) + hs)) & 3u);
        sc[j] = (int)(low | (high << 4)) - 32;
    }
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const LaneAct& X = act[i];
        const int bsum[4] = {lo16(X.bw[0]), hi16(X.bw[0]), lo16(X.bw[1]), hi16(X.bw[1])};
        const int xs[4][4] = {{X.x[0].x, X.x[0].y, X.x[0].z, X.x[0].w}, {X.x[1].x, X.x[1].y, X.x[1].z, X.x[1].w},
                              {X.x[2].x, X.x[2].y, X.x[2].z, X.x[2].w}, {X.x[3].x, X.x[3].y, X.x[3].z, X.x[3].w}};
        int isum = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int raw = 0;   // codes q3 + 4 in 0..7, so the exact dot is raw - 4 * bsum
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t c = ((qw[u] >> (2 * j)) & 0x03030303u) | (((hw[u] >> (4 * h + j)) & 0x01010101u) << 2);
                raw = dp4a_us(c, xs[j][u], raw);
            }
            const int dot = raw - 4 * bsum[j];
            if constexpr (SUBDOTS)
                sub_row[i * sub_stride_i + (size_t)b * 16 + 8 * h + 2 * j + p] = dot;
            isum += sc[j] * dot;
        }
        if constexpr (!SUBDOTS) v[i] = __fmaf_rn(__fmul_rn(d, X.dy), (float)isum, v[i]);
    }
}

// The per-lane block decode of format FMT (q2_K, q3_K, q6_K).
template <int FMT, int M, bool SUBDOTS>
__device__ __forceinline__ void fmt_block(const uint8_t* slot, int off, const LaneAct* act, int b, int t, float* v,
                                          int32_t* sub_row, size_t sub_stride_i) {
    if constexpr (FMT == 2)
        q2K_block<M, SUBDOTS>(slot, off, act, b, t, v, sub_row, sub_stride_i);
    else if constexpr (FMT == 3)
        q3K_block<M, SUBDOTS>(slot, off, act, b, t, v, sub_row, sub_stride_i);
    else
        q6K_block<M, SUBDOTS>(slot, off, act, b, t, v, sub_row, sub_stride_i);
}

// One block of the register path: adds this lane's f32 term of the block at
// byte offset off of the stage to v[] (same arithmetic as the staged path).
template <int FMT, int M>
__device__ __forceinline__ void areg_block(const uint8_t* slot, int off, const LaneAct* act, int t, float* v) {
    fmt_block<FMT, M, false>(slot, off, act, 0, t, v, nullptr, 0);
}

// AREG: each lane keeps the activations of its (at most two) block columns
// in registers for the whole segment; requires nb <= 16 and no SUBDOTS.
template <int FMT, int M, bool SUBDOTS, int WARPS, int MAXP, bool AREG>
__global__ void __launch_bounds__(WARPS * 32, 1) gemv_kernel(const __grid_constant__ GemvBatch<MAXP> B) {
    constexpr int SLOT = Fmt<FMT>::SLOT;
    constexpr int PAYLOAD = Fmt<FMT>::PAYLOAD;
    constexpr int BYTES = Fmt<FMT>::BYTES;
    static_assert(!(AREG && SUBDOTS), "register activations serve the f32 path only");
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int quad = lane >> 2, t = lane & 3;
    const int NS = B.nstages;
    uint8_t* ring = smem + B.act_bytes + (size_t)warp * NS * SLOT;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + B.act_bytes + (size_t)WARPS * NS * SLOT) + warp * NS;
    if (lane == 0) {
        for (int j = 0; j < NS; ++j) mbar_init(&bars[j], 1);
        fence_barrier_init();
    }
    __syncwarp();
    grid_launch_dependents();
    // without weight prefetch, nothing is touched before the earlier kernels end
    bool waited = !B.prefetch;
    if (waited) grid_wait_prior();

    const long long T = B.total_bytes;
    const long long B0 = T * blockIdx.x / gridDim.x;
    const long long B1 = T * (blockIdx.x + 1) / gridDim.x;
    uint32_t issued = 0, consumed = 0;   // ring counters, uniform in the warp
    uint32_t islot = 0, cslot = 0, cphase = 0;   // next slot to fill / to consume, its phase parity
    bool ok = true;                      // false once a wait ran out

    // problems are stored in byte order: start at the last one beginning at or before B0
    int pfirst = 0;
    for (int lo = 1, hi = B.count - 1; lo <= hi;) {
        const int mid = (lo + hi) >> 1;
        if (B.p[mid].byte_begin <= B0) { pfirst = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    for (int pi = pfirst; pi < B.count; ++pi) {
        const GemvProblem& P = B.p[pi];
        const long long rowbytes = (long long)P.nb * BYTES;
        const long long P0 = P.byte_begin;
        const long long P1 = P0 + (long long)P.n * rowbytes;
        if (P0 >= B1) break;                                      // CTA-uniform
        if (P1 <= B0) continue;
        // rows whose first byte falls in [B0, B1)
        const int ra = (int)ceil_div_ll(B0 > P0 ? B0 - P0 : 0, rowbytes);
        const long long rb_ll = ceil_div_ll(B1 - P0, rowbytes);
        const int rb = (int)(rb_ll < P.n ? rb_ll : P.n);
        if (ra >= rb) continue;                                    // CTA-uniform
        const int wa = ra + (int)((long long)(rb - ra) * warp / WARPS);
        const int wb = ra + (int)((long long)(rb - ra) * (warp + 1) / WARPS);
        const int nb = P.nb;
        const long long wbytes = (long long)P.n * rowbytes;
        const int rps = rowbytes <= PAYLOAD ? (int)(PAYLOAD / rowbytes) : 0;
        const int per_row = rps > 0 ? 1 : (nb + Fmt<FMT>::CHUNK - 1) / Fmt<FMT>::CHUNK;
        const int nst = wb > wa ? (rps > 0 ? (wb - wa + rps - 1) / rps : (wb - wa) * per_row) : 0;

        // issue cursor (uniform); lane 0 performs the copies
        int irow = wa, ib0 = 0, inext = 0;
        auto issue_one = [&]() {
            const StageGeom g = stage_geom<FMT>(irow, ib0, wb, rps, nb, wbytes);
            if (lane == 0) {
                uint64_t* bar = &bars[islot];
                uint8_t* dst = ring + islot * SLOT;
                if (g.bytes > 0) {
                    mbar_arrive_expect_tx(bar, (uint32_t)g.bytes);
                    bulk_g2s(dst, P.w + g.src, (uint32_t)g.bytes, bar);
                } else {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
                }
            }
            islot = islot + 1 == (uint32_t)NS ? 0 : islot + 1;
            ++issued;
            ++inext;
            if (rps > 0) {
                irow += rps;
            } else {
                ib0 += Fmt<FMT>::CHUNK;
                if (ib0 >= nb) { ib0 = 0; ++irow; }
            }
        };
        if (ok)
            while (inext < nst && issued - consumed < (uint32_t)NS) issue_one();

        if (!waited) {   // activations are read, and y written, only after the earlier kernels end
            grid_wait_prior();
            waited = true;
        }
        const bool packed = nb <= BLOCKS_PER_STEP && (BLOCKS_PER_STEP % nb) == 0;
        ActSmem act{};
        LaneAct areg[AREG ? 2 : 1][M];
        // register path geometry: packed rows -> row slot jrow, column quad % nb;
        // otherwise columns quad and quad + 8, clamped to the row (a clamped
        // column's result is discarded)
        const int jrow = packed ? quad / nb : 0;
        const int col0 = packed ? quad - jrow * nb : min(quad, nb - 1);
        const int col1 = min(quad + BLOCKS_PER_STEP, nb - 1);
        if constexpr (AREG) {
            if (nst > 0) {
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    areg[0][i] = act_from_global<FMT>(P.xq, i * nb + col0, t);
                    if (!packed) {
                        areg[1][i] = act_from_global<FMT>(P.xq, i * nb + col1, t);
                    }
                }
            }
        } else {
            __syncthreads();                   // every warp is done with the previous activations
            act = act_smem_carve(smem, M, nb);
            act_smem_fill<FMT>(act, P.xq, M, nb);
            __syncthreads();
        }

        const size_t sub_stride_i = (size_t)P.n * nb * Fmt<FMT>::SUB;
        float acc[M];
#pragma unroll
        for (int i = 0; i < M; ++i) acc[i] = 0.0f;
        int crow = wa, cb0 = 0;

        // processes block bb of row rr of the slot (activation column b)
        auto do_block = [&](uint8_t* slot, const StageGeom& g, int rr, int bb, int b, float* v,
                            int32_t* sub_row) {
            LaneAct la[M];
#pragma unroll
            for (int i = 0; i < M; ++i) la[i] = act_from_smem<FMT>(act, i * nb + b, t);
            fmt_block<FMT, M, SUBDOTS>(slot, g.delta + (rr * nb + bb) * BYTES, la, b, t, v, sub_row, sub_stride_i);
        };

        for (int s = 0; s < nst && ok; ++s) {
            if (!mbar_wait(&bars[cslot], cphase)) {
                // a copy never completed: record it, let our other copies land, stop computing
                if (lane == 0) {
                    atomicOr(B.fault, 1u);
                    for (uint32_t c2 = consumed; c2 < issued; ++c2) (void)mbar_wait(&bars[c2 % NS], (c2 / NS) & 1);
                }
                __syncwarp();
                ok = false;
                break;
            }
            uint8_t* slot = ring + cslot * SLOT;
            const StageGeom g = stage_geom<FMT>(crow, cb0, wb, rps, nb, wbytes);
            if (g.tail > 0) {   // the matrix's last bytes past its final 16-byte boundary
                if (lane < g.tail) slot[g.bytes + lane] = P.w[g.src + g.bytes + lane];
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            if constexpr (AREG) {
                const int nr = g.nrows;
                if (packed) {
                    // a step covers 8/nb whole rows (a row owns 4*nb lanes); two steps
                    // per iteration, rows past the stage clamped and not stored
                    constexpr int PU = 2;                  // steps per iteration
                    const int rw = BLOCKS_PER_STEP / nb;
                    for (int r0 = 0; r0 < nr; r0 += PU * rw) {
                        float v[PU][M];
#pragma unroll
                        for (int u = 0; u < PU; ++u) {
#pragma unroll
                            for (int i = 0; i < M; ++i) v[u][i] = 0.0f;
                            const int rr = min(r0 + jrow + u * rw, nr - 1);
                            areg_block<FMT, M>(slot, g.delta + (rr * nb + col0) * BYTES, areg[0], t, v[u]);
                        }
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) {
                            if (o <= 2 * nb) {
#pragma unroll
                                for (int u = 0; u < PU; ++u)
#pragma unroll
                                    for (int i = 0; i < M; ++i) v[u][i] += __shfl_xor_sync(0xFFFFFFFFu, v[u][i], o);
                            }
                        }
                        if ((lane & (4 * nb - 1)) == 0) {
#pragma unroll
                            for (int u = 0; u < PU; ++u) {
                                const int rr = r0 + jrow + u * rw;
#pragma unroll
                                for (int i = 0; i < M; ++i)
                                    if (rr < nr) P.y[(size_t)i * P.n + crow + rr] = v[u][i];
                            }
                        }
                    }
                } else {
                    // whole rows of at most 16 blocks: columns quad and quad + 8
                    const bool has0 = quad < nb, has1 = quad + BLOCKS_PER_STEP < nb;
                    // RU rows starting at stage row r0 (all below nr)
                    auto rows = [&](auto ru_tag, int r0) {
                        constexpr int RU = decltype(ru_tag)::value;
                        float v[RU][M];
#pragma unroll
                        for (int u = 0; u < RU; ++u) {
                            const int rr = r0 + u;
                            float a0[M], a1[M];
#pragma unroll
                            for (int i = 0; i < M; ++i) a0[i] = 0.0f;
                            areg_block<FMT, M>(slot, g.delta + (rr * nb + col0) * BYTES, areg[0], t, a0);
#pragma unroll
                            for (int i = 0; i < M; ++i) a1[i] = a0[i];
                            areg_block<FMT, M>(slot, g.delta + (rr * nb + col1) * BYTES, areg[1], t, a1);
#pragma unroll
                            for (int i = 0; i < M; ++i) v[u][i] = has1 ? a1[i] : (has0 ? a0[i] : 0.0f);
                        }
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
                            for (int u = 0; u < RU; ++u)
#pragma unroll
                                for (int i = 0; i < M; ++i) v[u][i] += __shfl_xor_sync(0xFFFFFFFFu, v[u][i], o);
                        }
                        if (lane == 0) {
#pragma unroll
                            for (int u = 0; u < RU; ++u)
#pragma unroll
                                for (int i = 0; i < M; ++i) P.y[(size_t)i * P.n + crow + r0 + u] = v[u][i];
                        }
                    };
                    int r0 = 0;
                    if constexpr (M == 1)
                        for (; r0 + 2 <= nr; r0 += 2) rows(std::integral_constant<int, 2>{}, r0);
                    for (; r0 < nr; ++r0) rows(std::integral_constant<int, 1>{}, r0);
                }
            } else if (packed) {
                // each step covers 8/nb whole rows; a row owns 4*nb lanes
                const int rpstep = BLOCKS_PER_STEP / nb;
                for (int r0 = 0; r0 < g.nrows; r0 += rpstep) {
                    const int rr = r0 + jrow;
                    const int row = crow + rr;
                    float v[M];
#pragma unroll
                    for (int i = 0; i < M; ++i) v[i] = 0.0f;
                    int32_t* sub_row = SUBDOTS ? P.sub + (size_t)row * nb * Fmt<FMT>::SUB : nullptr;
                    if (rr < g.nrows) do_block(slot, g, rr, col0, col0, v, sub_row);
                    if constexpr (!SUBDOTS) {
#pragma unroll
                        for (int i = 0; i < M; ++i) {
                            float x = v[i];
                            for (int o = 2 * nb; o >= 1; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
                            if ((lane & (4 * nb - 1)) == 0 && rr < g.nrows) P.y[(size_t)i * P.n + row] = x;
                        }
                    }
                }
            } else {
                for (int rr = 0; rr < g.nrows; ++rr) {
                    const int row = crow + rr;
                    int32_t* sub_row = SUBDOTS ? P.sub + (size_t)row * nb * Fmt<FMT>::SUB : nullptr;
                    for (int bb = quad; bb < g.nblk; bb += BLOCKS_PER_STEP)
                        do_block(slot, g, rr, bb, cb0 + bb, acc, sub_row);
                    const bool row_end = rps > 0 || cb0 + g.nblk >= nb;
                    if (row_end) {
                        if constexpr (!SUBDOTS) {
#pragma unroll
                            for (int i = 0; i < M; ++i) {
                                const float x = warp_sum(acc[i]);
                                if (lane == 0) P.y[(size_t)i * P.n + row] = x;
                                acc[i] = 0.0f;
                            }
                        }
                    }
                }
            }
            ++consumed;
            if (++cslot == (uint32_t)NS) {
                cslot = 0;
                cphase ^= 1u;
            }
            if (rps > 0) {
                crow += rps;
            } else {
                cb0 += Fmt<FMT>::CHUNK;
                if (cb0 >= nb) { cb0 = 0; ++crow; }
            }
            __syncwarp();
            if (inext < nst) issue_one();
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
inline int smem_optin_bytes() {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return optin;
}

inline size_t act_bytes_aligned(int m, int nb) { return (act_smem_bytes(m, nb) + 127) & ~(size_t)127; }

template <int FMT>
inline int ring_depth(int m, int nb, int warps) {
    const long long budget = (long long)smem_optin_bytes() - (long long)act_bytes_aligned(m, nb);
    const long long per_stage = (long long)warps * (Fmt<FMT>::SLOT + 8);
    long long ns = budget / per_stage;
    if (ns > MAX_STAGES) ns = MAX_STAGES;
    return ns >= 2 ? (int)ns : 0;
}

template <int FMT>
inline size_t gemv_smem(int m, int nb, int ns, int warps) {
    return act_bytes_aligned(m, nb) + (size_t)warps * ns * (Fmt<FMT>::SLOT + 8);
}

struct HostProblem {
    const uint8_t* w;
    const uint8_t* xq;
    float* y;
    int32_t* sub;
    int n, nb;
    const uint8_t* w2 = nullptr;   // paired q4_K launches: the up matrix
};

template <int FMT, int M, bool SUB, int WARPS, int MAXP, bool AREG>
cudaError_t launch_batch(const HostProblem* hp, int count, int max_nb, int ns, cudaStream_t stream) {
    GemvBatch<MAXP> B;
    B.fault = fault_word();
    if (!B.fault) return cudaErrorInvalidDevicePointer;
    long long off = 0, rows = 0;
    for (int i = 0; i < count; ++i) {
        B.p[i].w = hp[i].w;
        B.p[i].xq = hp[i].xq;
        B.p[i].y = hp[i].y;
        B.p[i].sub = hp[i].sub;
        B.p[i].byte_begin = off;
        B.p[i].n = hp[i].n;
        B.p[i].nb = hp[i].nb;
        off += (long long)hp[i].n * hp[i].nb * Fmt<FMT>::BYTES;
        rows += hp[i].n;
    }
    B.total_bytes = off;
    B.count = count;
    B.nstages = ns;
    B.act_bytes = AREG ? 0 : (int)act_bytes_aligned(M, max_nb);
    const size_t smem = (size_t)B.act_bytes + (size_t)WARPS * ns * (Fmt<FMT>::SLOT + 8);
    const void* fn = (const void*)gemv_kernel<FMT, M, SUB, WARPS, MAXP, AREG>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    long long grid = num_sms();
    const long long want = (rows + 7) / 8;
    if (grid > want) grid = want;
    if (grid < 1) grid = 1;
    B.prefetch = overlap_mode() >= 2 ? 1 : 0;
    return launch_kernel(gemv_kernel<FMT, M, SUB, WARPS, MAXP, AREG>, dim3((unsigned)grid), dim3(WARPS * 32), smem,
                         stream, B);
}

// Launches one pass (all problems share m = M rows of activations).
template <int FMT, int M, bool SUB>
cudaError_t launch_pass(const HostProblem* hp, int count, int max_nb, cudaStream_t stream) {
    if constexpr (!SUB && M <= 1) {
        // activations in registers: rows of at most 16 blocks (q6_K: m = 1 only,
        // the register budget of two activation rows is exceeded)
        if (max_nb <= 16) {
            const int ns = ring_depth<FMT>(0, max_nb, GEMV_WARPS);
            if (count == 1) return launch_batch<FMT, M, SUB, GEMV_WARPS, 1, true>(hp, count, max_nb, ns, stream);
            return launch_batch<FMT, M, SUB, GEMV_WARPS, GROUP_MAX, true>(hp, count, max_nb, ns, stream);
        }
    }
    const int ns = ring_depth<FMT>(M, max_nb, GEMV_WARPS);
    if (ns < 2) return cudaErrorInvalidConfiguration;
    if constexpr (SUB) {
        return launch_batch<FMT, M, SUB, GEMV_WARPS, 1, false>(hp, count, max_nb, ns, stream);
    } else {
        if (count == 1) return launch_batch<FMT, M, SUB, GEMV_WARPS, 1, false>(hp, count, max_nb, ns, stream);
        return launch_batch<FMT, M, SUB, GEMV_WARPS, GROUP_MAX, false>(hp, count, max_nb, ns, stream);
    }
}

template <int FMT, bool SUB>
cudaError_t dispatch_m(int m, const HostProblem* hp, int count, int max_nb, cudaStream_t stream) {
    switch (m) {
        case 1: return launch_pass<FMT, 1, SUB>(hp, count, max_nb, stream);
        case 2: return launch_pass<FMT, 2, SUB>(hp, count, max_nb, stream);
        case 3: return launch_pass<FMT, 3, SUB>(hp, count, max_nb, stream);
        case 4: return launch_pass<FMT, 4, SUB>(hp, count, max_nb, stream);
        case 5: return launch_pass<FMT, 5, SUB>(hp, count, max_nb, stream);
        case 6: return launch_pass<FMT, 6, SUB>(hp, count, max_nb, stream);
        case 7: return launch_pass<FMT, 7, SUB>(hp, count, max_nb, stream);
        case 8: return launch_pass<FMT, 8, SUB>(hp, count, max_nb, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Rows of activations per pass so that the staged activations leave room
// for a ring of at least two stages (16 warps).  The work split and the f32
// order of a row do not depend on m, so splitting m changes no bits.
template <int FMT>
int gemv_rows_per_pass(int m, int max_nb) {
    int step = m;
    while (step > 1 && ring_depth<FMT>(step, max_nb, GEMV_WARPS) == 0) --step;
    return ring_depth<FMT>(step, max_nb, GEMV_WARPS) ? step : 0;
}

// Runs a group of problems with m activation rows each (1 <= m <= 8),
// taking the activation rows in passes and the problems GROUP_MAX at a time.
template <int FMT>
cudaError_t run_group(const HostProblem* probs, int count, int m, bool subdots, cudaStream_t stream) {
    int max_nb = 1;
    for (int i = 0; i < count; ++i) max_nb = probs[i].nb > max_nb ? probs[i].nb : max_nb;
    const int step = gemv_rows_per_pass<FMT>(m, max_nb);
    if (step < 1) return cudaErrorInvalidConfiguration;
    HostProblem part[GROUP_MAX];
    for (int i0 = 0; i0 < m; i0 += step) {
        const int mm = m - i0 < step ? m - i0 : step;
        for (int p0 = 0; p0 < count; p0 += GROUP_MAX) {
            const int cnt = count - p0 < GROUP_MAX ? count - p0 : GROUP_MAX;
            int pnb = 1;
            for (int j = 0; j < cnt; ++j) {
                const HostProblem& s = probs[p0 + j];
                part[j] = s;
                part[j].xq = s.xq + (size_t)i0 * s.nb * Q8K_BYTES;
                part[j].y = s.y ? s.y + (size_t)i0 * s.n : nullptr;
                part[j].sub = s.sub ? s.sub + (size_t)i0 * s.n * s.nb * Fmt<FMT>::SUB : nullptr;
                pnb = s.nb > pnb ? s.nb : pnb;
            }
            const cudaError_t e = subdots ? dispatch_m<FMT, true>(mm, part, cnt, pnb, stream)
                                          : dispatch_m<FMT, false>(mm, part, cnt, pnb, stream);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace plm
