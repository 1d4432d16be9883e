// Decode GEMV for m = 1..8 activation rows on the tensor cores, over the
// row-interleaved q4_K layout "x16" (PocketLLM, Korean README, "Current
// status" table, row "src/": the packed q4_K dot gains from an 8-column
// panel repack of the weights and an 8-row activation tile; here the repack
// interleaves 16 weight rows per 256-weight block and the activation tile is
// the m <= 8 columns of an MMA).
//
// Layout x16 (same bytes as the GGML q4_K blocks, 16-byte units permuted):
// rows are grouped in tiles of 16 (the last tile padded with zero blocks);
// tile-block (T, b) -- rows 16T..16T+15, block b -- is 2304 contiguous bytes
// at ((T * nb) + b) * 2304:
//   [0, 256)      the 16-byte headers (f16 d, f16 dmin, scales[12]) of rows
//                 16T + 0 .. 16T + 15, row r at 16 r;
//   [256, 2304)   qs: for j = 0..3 and lane L = 0..31 (g = L / 4, t = L % 4),
//                 offset 256 + 512 j + 16 L holds 16 qs bytes: j = 0, 1: row
//                 g, qs[32t + 16j ..]; j = 2, 3: row g + 8, qs[32t + 16(j-2) ..].
// So a tile's blocks stream as one contiguous run, and lane L of a warp reads
// exactly its own 64 qs bytes with four 16-byte loads that are contiguous
// across the warp.
//
// Arithmetic.  Per 256-weight block and 16-row tile, one warp runs sixteen
// mma.sync.m16n8k16 (f16 operands, f32 accumulation): A = the decoded
// weights sc_j * q (integers <= 945, exact in f16), B = the q8 activation
// codes of up to eight activation rows (exact in f16), so each MMA adds exact
// integer products; a 17th MMA forms the min term sum_j m_j * (bsum_2j +
// bsum_2j+1) from the six-bit mins and the bsums.  The block's f32 term
// d_x * (d * isum - dmin * msum) is applied per output element, the same
// arithmetic as the other kernels.  Lane (g, t) holds rows g, g + 8 of the
// tile and the 64 weights of chunk t; MMA kk = 2u + s takes, at A positions
// 2t + e, the low nibbles of bytes s and 2 + s of qs word u (weights
// 64t + 4u + 2e + s) and at positions 2t + 8 + e the high nibbles (the same
// weights + 32); the activation fragments use the same permutation of k.  In
// the min MMA, lane t's positions 2t, 2t + 1, 2t + 8, 2t + 9 carry the bsum
// groups 4t .. 4t + 3, i.e. sub-blocks 2t and 2t + 1, whose scales the lane
// already holds.  The decode is the magic-number form: (1024 + q) * sc -
// 1024 * sc and (1024 + 16 q) * sc / 16 - 64 sc in one hfma2, exact for every
// code.
//
// Work split: a persistent grid, one CTA of 16 warps per SM.  CTA c takes
// tiles [T c / G, T (c + 1) / G).  Its warps form TEAMS teams of KW warps
// (KW the largest power of two <= 16 dividing nb); warp kw of a team takes
// blocks [kw * nb / KW, (kw + 1) * nb / KW) of each of the team's tiles and
// keeps the activation fragments of one block in registers.  Tiles are taken
// in rounds of six per team; after a round the KW partial sums of every
// tile are added in kw order through shared memory (so the f32 order depends
// only on nb, never on m) and y is written.  Each warp streams its
// tile-blocks through a private ring of bulk copies with bounded waits.
#include "gemv_impl.cuh"

namespace plm {
namespace x16 {

constexpr int TR = 16;                      // weight rows per tile (MMA M)
// bytes of one tile-block (16 rows x one 256-weight block)
template <int FMT> struct X16;
// and the ring slots per warp that fit beside the partial sums
template <> struct X16<4> { static constexpr int TB = TR * Q4K_BYTES, NS = 4; };   // 2304
template <> struct X16<6> { static constexpr int TB = TR * Q6K_BYTES, NS = 3; };   // 3360
constexpr int WARPS = 16;
constexpr int THREADS = WARPS * 32;
constexpr int R = 6;                        // tiles per team per round
constexpr int PSTRIDE = 20;                 // floats per activation row of a partial tile (16 rows + pad)
constexpr int PART_FLOATS = 8 * PSTRIDE;    // one warp's partial sums of one tile: [col][row], padded
constexpr int PART_BYTES = WARPS * R * PART_FLOATS * 4;   // 60 KB of partial sums per round
template <int FMT> __host__ __device__ constexpr int ring_bytes() { return WARPS * X16<FMT>::NS * X16<FMT>::TB; }
template <int FMT> __host__ __device__ constexpr int smem_bytes() {
    return PART_BYTES + ring_bytes<FMT>() + WARPS * X16<FMT>::NS * 8;
}
static_assert(smem_bytes<4>() <= 227 * 1024 && smem_bytes<6>() <= 227 * 1024, "x16 shared memory");

struct Args {
    const uint8_t* w;        // x16 tile-blocks [ntiles][nb]
    const uint8_t* xq;       // q8_K [m][nb]
    float* y;                // [m][n]
    unsigned* fault;
    int m, n, nb, ntiles;
    int kw_log2;             // KW = 1 << kw_log2 warps per team
    int prefetch;            // copy weights before waiting for the kernels before this one
    // decode constants passed as values, so that they stay in registers
    // (0x000F000F, 0x00F000F0, 0x64006400, 1 << 24)
    uint32_t kmlo, kmhi, kmagic, k2p24;
    uint32_t km1056;         // f16 pair (-1056, -1056)
    uint32_t k0f, k30;       // 0x0F0F0F0F, 0x30303030
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two signed activation codes (bytes 0 and 2 of p, zero-extended) as an
// exact f16 pair: 1024 + 128 + x through the bit pattern, minus 1152.
__device__ __forceinline__ uint32_t codes_to_h2(uint32_t p) {
    const uint32_t v = (p ^ 0x00800080u) | 0x64006400u;   // once per block and kernel: not on the hot path
    return h2u(__hsub2(u2h(v), u2h(0x64806480u)));
}

// Activation fragments of one 256-value block for lane (g, t): row g of the
// activations (zero when g >= m) in the kernel's k order; q4_K: the weights
// of chunk t and the min term's bsum fragment; q6_K: values 16G + 4t ..
// 16G + 4t + 3 of every 16-group G.  And d of activation rows 2t, 2t + 1.
struct BFrag {
    uint32_t b[16][2];
    uint32_t bm[2];
    float dx[2];
};

template <int FMT>
__device__ __forceinline__ void load_bfrag(BFrag& F, const uint8_t* __restrict__ xq, int m, int nb, int b, int g,
                                           int t) {
    if (FMT == 6 && g < m) {
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(xq + ((size_t)g * nb + b) * Q8K_BYTES + 4) + t;
#pragma unroll
        for (int G = 0; G < 16; ++G) {
            const uint32_t x = __ldg(cw + 4 * G);
            F.b[G][0] = codes_to_h2(__byte_perm(x, 0, 0x4140));
            F.b[G][1] = codes_to_h2(__byte_perm(x, 0, 0x4342));
        }
        F.bm[0] = F.bm[1] = 0u;
    } else if (FMT == 4 && g < m) {
        const uint8_t* blk = xq + ((size_t)g * nb + b) * Q8K_BYTES;
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(blk + 4 + 64 * t);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t x0 = __ldg(cw + u), x1 = __ldg(cw + 8 + u);
            F.b[2 * u][0] = codes_to_h2(__byte_perm(x0, 0, 0x4240));
            F.b[2 * u][1] = codes_to_h2(__byte_perm(x1, 0, 0x4240));
            F.b[2 * u + 1][0] = codes_to_h2(__byte_perm(x0, 0, 0x4341));
            F.b[2 * u + 1][1] = codes_to_h2(__byte_perm(x1, 0, 0x4341));
        }
        const uint32_t* bw = reinterpret_cast<const uint32_t*>(blk + 260);
        const uint32_t s0 = __ldg(bw + 2 * t), s1 = __ldg(bw + 2 * t + 1);   // bsums (4t, 4t+1), (4t+2, 4t+3)
        F.bm[0] = h2u(__halves2half2(__short2half_rn((short)(s0 & 0xFFFF)), __short2half_rn((short)(s0 >> 16))));
        F.bm[1] = h2u(__halves2half2(__short2half_rn((short)(s1 & 0xFFFF)), __short2half_rn((short)(s1 >> 16))));
    } else {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) F.b[kk][0] = F.b[kk][1] = 0u;
        F.bm[0] = F.bm[1] = 0u;
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int row = 2 * t + c;
        F.dx[c] = row < m ? __ldg(reinterpret_cast<const float*>(xq + ((size_t)row * nb + b) * Q8K_BYTES)) : 0.0f;
    }
}

// Per-row constants of one block for lane t: the f16 pairs that decode the
// low nibbles (sub-block 2t) and high nibbles (sub-block 2t + 1), the mins
// m_2t, m_(2t+1) as the min term's A fragment, and d, dmin.
struct RowC {
    uint32_t slo, olo, shi, ohi, mlo, mhi;
    float d, dmin;
};

// Sub-blocks 2t, 2t + 1 of the 12-byte table (scale bytes s[0..11] = words
// Y, Z, W): t < 2: sc = s[j] & 63, m = s[j + 4] & 63; t >= 2 (j = 2t - 4 +
// {0, 1}): sc = (s[j + 8] & 15) | (s[j] >> 6) << 4, m = (s[j + 8] >> 4) |
// (s[j + 4] >> 6) << 4.  The lane's shifts and masks pick its case.
struct LaneC {
    uint32_t shs, shm, hsh;       // shift of the low part of sc / m, shift of the top-bit source
    uint32_t mask1, mask2;        // low-part mask, top-bit mask
    bool lowpair;                 // t < 2
};

__device__ __forceinline__ RowC row_consts(const uint4 h, const LaneC& L) {
    RowC R;
    const __half2 dd = u2h(h.x);
    R.d = __low2float(dd);
    R.dmin = __high2float(dd);
    // sc_2t, sc_(2t+1) in bytes 0, 1; m_2t, m_(2t+1) in bytes 0, 1
    const uint32_t ss = L.lowpair ? h.y : h.w, sm = L.lowpair ? h.z : h.w;
    const uint32_t sc = ((ss >> L.shs) & L.mask1) | ((h.y >> L.hsh) & L.mask2);
    const uint32_t mm = ((sm >> L.shm) & L.mask1) | ((h.z >> L.hsh) & L.mask2);
    const __half2 k1024 = u2h(0x64006400u);
    const __half2 s0 = __hsub2(u2h(__byte_perm(sc, 0x64, 0x4040)), k1024);
    const __half2 s1 = __hsub2(u2h(__byte_perm(sc, 0x64, 0x4141)), k1024);
    R.slo = h2u(s0);
    R.olo = h2u(__hmul2(s0, u2h(0xE400E400u)));   // x (-1024)
    R.shi = h2u(__hmul2(s1, u2h(0x2C002C00u)));   // x 1/16
    R.ohi = h2u(__hmul2(s1, u2h(0xD400D400u)));   // x (-64)
    R.mlo = h2u(__hsub2(u2h(__byte_perm(mm, 0x64, 0x4040)), k1024));
    R.mhi = h2u(__hsub2(u2h(__byte_perm(mm, 0x64, 0x4141)), k1024));
    return R;
}

// (a & b) | c in one instruction (b and c in registers, so that the
// compiler does not split the two constants over two operations)
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Decode constants held in registers for the whole kernel.
struct DecK {
    uint32_t mlo, mhi, magic;   // 0x000F000F, 0x00F000F0, 0x64006400
    uint32_t p24;               // 1 << 24: w >> 8 as a multiply-high (the integer-multiply pipe)
};

__device__ __forceinline__ uint32_t dec(uint32_t w, uint32_t mask, uint32_t magic, uint32_t s, uint32_t o) {
    return h2u(__hfma2(u2h(and_or(w, mask, magic)), u2h(s), u2h(o)));
}

// One tile-block: the f32 terms of rows g, g + 8 and activation rows 2t,
// 2t + 1, added to acc[0..3].  The sixteen main MMAs run as two independent
// accumulator chains (even and odd kk) that are added at the end: every
// partial sum is an exact integer below 2^24 except for adversarial blocks,
// and the order is fixed, so the result depends on nothing but the data.
__device__ __forceinline__ void tile_block(const uint8_t* slot, int g, int lane, const LaneC& L, const DecK& K,
                                           const BFrag& F, float (&acc)[4]) {
    const uint4 hg = *reinterpret_cast<const uint4*>(slot + 16 * g);
    const uint4 hh = *reinterpret_cast<const uint4*>(slot + 16 * (g + 8));
    const uint4* qp = reinterpret_cast<const uint4*>(slot + 256) + lane;
    const uint4 q0 = qp[0], q1 = qp[32], q2 = qp[64], q3 = qp[96];
    const RowC G = row_consts(hg, L), H = row_consts(hh, L);
    const uint32_t wg[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t wh[8] = {q2.x, q2.y, q2.z, q2.w, q3.x, q3.y, q3.z, q3.w};
    float ce[4] = {0.f, 0.f, 0.f, 0.f}, co[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t a = wg[u], b = wh[u], a1 = __umulhi(a, K.p24), b1 = __umulhi(b, K.p24);
        mma16816(ce, dec(a, K.mlo, K.magic, G.slo, G.olo), dec(b, K.mlo, K.magic, H.slo, H.olo),
                 dec(a, K.mhi, K.magic, G.shi, G.ohi), dec(b, K.mhi, K.magic, H.shi, H.ohi), F.b[2 * u][0],
                 F.b[2 * u][1]);
        mma16816(co, dec(a1, K.mlo, K.magic, G.slo, G.olo), dec(b1, K.mlo, K.magic, H.slo, H.olo),
                 dec(a1, K.mhi, K.magic, G.shi, G.ohi), dec(b1, K.mhi, K.magic, H.shi, H.ohi), F.b[2 * u + 1][0],
                 F.b[2 * u + 1][1]);
    }
    mma16816(c2, G.mlo, H.mlo, G.mhi, H.mhi, F.bm[0], F.bm[1]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float d = j < 2 ? G.d : H.d, dm = j < 2 ? G.dmin : H.dmin;
        const float term = __fmaf_rn(d, __fadd_rn(ce[j], co[j]), -__fmul_rn(dm, c2[j]));
        acc[j] = __fmaf_rn(F.dx[j & 1], term, acc[j]);
    }
}

// q6_K tile-block (x16 layout, 3360 bytes): [0, 256) the int8 scales of the
// 16 rows (row i at 16 i); [256, 288) their f16 d; [288, 2336) ql: for
// j = 0..3 and lane L = (g, t), 16 bytes at 288 + 512 j + 16 L holding the
// 4-byte pieces ql[64h + 16w + 4t ..] (w = 0..3, h = j % 2) of row g (j < 2)
// or g + 8; [2336, 3360) qh: for j = 0..1, 16 bytes at 2336 + 512 j + 16 L
// holding qh[32h + 16s + 4t ..] for (h, s) = (0,0), (0,1), (1,0), (1,1) of row
// g + 8 j.  One MMA per 16-group G = 8h + 2qq + s: lane t's A positions
// 2t + e and 2t + 8 + e carry the codes of weights 16G + 4t + e and
// 16G + 4t + 2 + e as the exact f16 values q6 - 32; the group's int8 scale
// is applied to the MMA's exact integer result in f32 (sc * D < 2^24), so
// every int8 scale is exact.
struct Q6Consts {
    uint32_t k0f, k30, magic, m1056;   // 0x0F0F0F0F, 0x30303030, 0x64, f16 (-1056, -1056)
};

// Signed byte b of w as f32, by the integer-to-float conversion (exact)
__device__ __forceinline__ float sbyte_i2f(uint32_t w, int b) {
    return __int2float_rn((int)(int8_t)(uint8_t)(w >> (8 * b)));
}

__device__ __forceinline__ void tile_block_q6(const uint8_t* slot, int g, int lane, const Q6Consts& K,
                                              const BFrag& F, float (&acc)[4]) {
    const uint4 sg = *reinterpret_cast<const uint4*>(slot + 16 * g);
    const uint4 sh = *reinterpret_cast<const uint4*>(slot + 16 * (g + 8));
    const float dg = __half2float(*reinterpret_cast<const __half*>(slot + 256 + 2 * g));
    const float dh = __half2float(*reinterpret_cast<const __half*>(slot + 256 + 2 * (g + 8)));
    const uint4* lp = reinterpret_cast<const uint4*>(slot + 288) + lane;
    const uint4 l0 = lp[0], l1 = lp[32], l2 = lp[64], l3 = lp[96];
    const uint4* hp = reinterpret_cast<const uint4*>(slot + 2336) + lane;
    const uint4 h0 = hp[0], h1 = hp[32];
    const uint32_t qlg[2][4] = {{l0.x, l0.y, l0.z, l0.w}, {l1.x, l1.y, l1.z, l1.w}};
    const uint32_t qlh[2][4] = {{l2.x, l2.y, l2.z, l2.w}, {l3.x, l3.y, l3.z, l3.w}};
    const uint32_t qhg[4] = {h0.x, h0.y, h0.z, h0.w}, qhh[4] = {h1.x, h1.y, h1.z, h1.w};
    const uint32_t scg[4] = {sg.x, sg.y, sg.z, sg.w};
    const uint32_t sch[4] = {sh.x, sh.y, sh.z, sh.w};
    float is[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const uint32_t hg = qhg[2 * h + s], hh = qhh[2 * h + s];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const int G = 8 * h + 2 * qq + s;
                // top two bits of each code (bits 2qq, 2qq + 1 of qh) to bits 4-5
                const uint32_t tg = (qq < 2 ? hg << (4 - 2 * qq) : hg >> (2 * qq - 4)) & K.k30;
                const uint32_t th = (qq < 2 ? hh << (4 - 2 * qq) : hh >> (2 * qq - 4)) & K.k30;
                // low four bits: low nibbles of ql for quarters 0, 1, high nibbles for 2, 3
                const uint32_t lg = qlg[h][2 * (qq & 1) + s], lh = qlh[h][2 * (qq & 1) + s];
                const uint32_t cg = and_or(qq < 2 ? lg : lg >> 4, K.k0f, tg);
                const uint32_t ch = and_or(qq < 2 ? lh : lh >> 4, K.k0f, th);
                // (1024 + q6) pairs through the bit pattern, minus 1056: q6 - 32, exact
                const __half2 m1056 = u2h(K.m1056);
                const uint32_t a0 = h2u(__hadd2(u2h(__byte_perm(cg, K.magic, 0x4140)), m1056));
                const uint32_t a1 = h2u(__hadd2(u2h(__byte_perm(ch, K.magic, 0x4140)), m1056));
                const uint32_t a2 = h2u(__hadd2(u2h(__byte_perm(cg, K.magic, 0x4342)), m1056));
                const uint32_t a3 = h2u(__hadd2(u2h(__byte_perm(ch, K.magic, 0x4342)), m1056));
                float dd[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(dd, a0, a1, a2, a3, F.b[G][0], F.b[G][1]);
                const float s_g = sbyte_i2f(scg[G >> 2], G & 3), s_h = sbyte_i2f(sch[G >> 2], G & 3);
                is[0] = __fmaf_rn(s_g, dd[0], is[0]);
                is[1] = __fmaf_rn(s_g, dd[1], is[1]);
                is[2] = __fmaf_rn(s_h, dd[2], is[2]);
                is[3] = __fmaf_rn(s_h, dd[3], is[3]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = __fmaf_rn(F.dx[j & 1], __fmul_rn(j < 2 ? dg : dh, is[j]), acc[j]);
}

template <int FMT>
__global__ void __launch_bounds__(THREADS, 1) gemv_x16_kernel(const __grid_constant__ Args A) {
    constexpr int TB = X16<FMT>::TB, NS = X16<FMT>::NS;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    float* part = reinterpret_cast<float*>(smem);
    uint8_t* ring = smem + PART_BYTES + (size_t)warp * NS * TB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PART_BYTES + ring_bytes<FMT>()) + warp * NS;
    if (lane == 0) {
        for (int j = 0; j < NS; ++j) mbar_init(&bars[j], 1);
        fence_barrier_init();
    }
    __syncwarp();
    grid_launch_dependents();

    // KW and TEAMS are powers of two: every index below is a shift or a mask
    const int kl = A.kw_log2, tl = 4 - kl;
    const int KW = 1 << kl, TEAMS = 1 << tl;
    const int team = warp >> kl, kw = warp & (KW - 1);
    const int nb = A.nb, BPW = nb >> kl;
    const int ct0 = (int)((long long)A.ntiles * blockIdx.x / gridDim.x);
    const int ct1 = (int)((long long)A.ntiles * (blockIdx.x + 1) / gridDim.x);
    const int ntc = ct1 - ct0, RT = R << tl;
    // tiles of this warp's team in the round starting at rb (tile rb + team + TEAMS * ti)
    auto tiles_in = [&](int rb) { return min(R, max(0, (ntc - rb - team + TEAMS - 1) >> tl)); };

    // copy cursor: the warp's tile-blocks in consumption order (round, then
    // block, then tile); lane 0 issues the copies
    const uint8_t* wbase = A.w + ((size_t)(ct0 + team) * nb + kw * BPW) * TB;
    const size_t tstride = ((size_t)nb * TB) << tl;   // next tile of the team
    int irb = 0, ibi = 0, iti = 0, icnt = tiles_in(0);
    const uint8_t* isrc = wbase;   // (irb, ibi, iti = 0)
    uint32_t issued = 0, islot = 0;
    auto issue_all = [&](uint32_t consumed) {
        while (irb < ntc && issued - consumed < (uint32_t)NS) {
            while (iti >= icnt) {   // next block of the round, or the next round
                iti = 0;
                if (icnt == 0 || ++ibi >= BPW) {
                    ibi = 0;
                    irb += RT;
                    if (irb >= ntc) return;   // irb >= ntc: nothing is issued again
                    icnt = tiles_in(irb);
                }
                isrc = wbase + (size_t)irb * ((size_t)nb * TB) + (size_t)ibi * TB;
            }
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the slot's reads before the refill
                mbar_arrive_expect_tx(&bars[islot], TB);
                bulk_g2s(ring + islot * TB, isrc, TB, &bars[islot]);
            }
            isrc += tstride;
            islot = islot + 1 == NS ? 0 : islot + 1;
            ++issued;
            ++iti;
        }
    };
    if (A.prefetch) issue_all(0);
    grid_wait_prior();   // activations are read and y written only after the earlier kernels end
    issue_all(0);

    LaneC L;
    L.lowpair = t < 2;
    const uint32_t h16 = 16u * (t & 1);
    L.shs = h16;
    L.shm = L.lowpair ? h16 : h16 + 4;
    L.hsh = h16 + 2;
    L.mask1 = L.lowpair ? 0x3F3Fu : 0x0F0Fu;
    L.mask2 = L.lowpair ? 0u : 0x3030u;
    DecK K;
    K.mlo = A.kmlo;
    K.mhi = A.kmhi;
    K.magic = A.kmagic;
    K.p24 = A.k2p24;
    Q6Consts K6;
    K6.k0f = A.k0f;
    K6.k30 = A.k30;
    K6.magic = A.kmagic >> 24;               // 0x64
    K6.m1056 = A.km1056;

    uint32_t consumed = 0, cslot = 0, cphase = 0;
    bool ok = true;
    BFrag F;
    int fbk = -1;   // block whose fragments F holds
    for (int rb = 0; rb < ntc; rb += RT) {
        const int nt = tiles_in(rb);
        // this lane's partials of tile 0: [col][row] with a padded row stride,
        // so the four stores of a warp touch 32 distinct banks
        float* pw = part + ((size_t)team * R * KW + kw) * PART_FLOATS + 2 * t * PSTRIDE + g;
        for (int bi = 0; bi < BPW && nt > 0 && ok; ++bi) {
            const int b = kw * BPW + bi;
            if (b != fbk) {
                load_bfrag<FMT>(F, A.xq, A.m, nb, b, g, t);
                fbk = b;
            }
#pragma unroll 1
            for (int ti = 0; ti < nt; ++ti) {
                if (!mbar_wait(&bars[cslot], cphase)) {
                    // a copy never landed: record it and stop (the round's
                    // barriers are still kept, so the CTA does not hang)
                    ok = false;
                    if (lane == 0) atomicOr(A.fault, 1u);
                    break;
                }
                // acc[0..3]: (row g, col 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
                float* pp = pw + (size_t)ti * KW * PART_FLOATS;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (bi > 0) {
                    acc[0] = pp[0];
                    acc[1] = pp[PSTRIDE];
                    acc[2] = pp[8];
                    acc[3] = pp[PSTRIDE + 8];
                }
                if constexpr (FMT == 4)
                    tile_block(ring + cslot * TB, g, lane, L, K, F, acc);
                else
                    tile_block_q6(ring + cslot * TB, g, lane, K6, F, acc);
                pp[0] = acc[0];
                pp[PSTRIDE] = acc[1];
                pp[8] = acc[2];
                pp[PSTRIDE + 8] = acc[3];
                __syncwarp();
                ++consumed;
                if (++cslot == NS) { cslot = 0; cphase ^= 1u; }
                issue_all(consumed);
            }
        }
        __syncthreads();
        // y for the round's tiles, all m activation rows at once (the other warps
        // wait meanwhile): item i is activation row col = i / nout and tile row
        // r = i % nout, i.e. (tile slot j, row) = (r / 16, r % 16); its KW
        // partials are loaded together and added in kw order
        const int nout = min(RT, ntc - rb) * TR;
        for (int i = threadIdx.x; i < A.m * nout; i += THREADS) {
            const int col = i / nout, r = i - col * nout;
            const int j = r >> 4, row = r & 15;
            const int grow = (ct0 + rb + j) * TR + row;
            if (grow < A.n) {
                const float* pp =
                    part + ((size_t)((j & (TEAMS - 1)) * R + (j >> tl)) * KW) * PART_FLOATS + col * PSTRIDE + row;
                float sum = pp[0];
#pragma unroll
                for (int q0 = 0; q0 < WARPS; q0 += 8) {   // eight loads in flight, then their adds
                    float v[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[q] = q0 + q < KW ? pp[(q0 + q) * PART_FLOATS] : 0.0f;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (q0 + q >= 1 && q0 + q < KW) sum += v[q];
                }
                A.y[(size_t)col * A.n + grow] = sum;
            }
        }
        __syncthreads();
    }
    // after a wait ran out: let this warp's copies still in flight (from the
    // one that did not land on) land before the CTA exits
    if (!ok && lane == 0)
        for (uint32_t c = consumed; c < issued; ++c) (void)mbar_wait(&bars[c % NS], (c / NS) & 1u);
}

// x16 repack of q4_K: one thread per 16-byte unit of the output.
__global__ void repack_x16_q4K_kernel(const uint8_t* __restrict__ w, uint8_t* __restrict__ out, int n, int nb,
                                      long long units) {
    grid_launch_dependents();
    grid_wait_prior();
    constexpr int UPB = X16<4>::TB / 16;   // 144 units per tile-block
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        const long long tb = u / UPB;
        const int o = (int)(u - tb * UPB);
        const long long tile = tb / nb;
        const int b = (int)(tb - tile * nb);
        int row, src;
        if (o < 16) {
            row = o;
            src = 0;
        } else {
            const int j = (o - 16) >> 5, L = (o - 16) & 31;
            row = (L >> 2) + (j >= 2 ? 8 : 0);
            src = 16 + 32 * (L & 3) + 16 * (j & 1);
        }
        const long long r = tile * TR + row;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < n) v = *reinterpret_cast<const uint4*>(w + ((size_t)r * nb + b) * Q4K_BYTES + src);
        reinterpret_cast<uint4*>(out)[u] = v;
    }
}

// x16 repack of q6_K: one thread per 16-byte unit of the output, gathered as
// four 4-byte pieces (q6_K blocks are only 2-byte aligned: 16-bit loads).
__global__ void repack_x16_q6K_kernel(const uint8_t* __restrict__ w, uint8_t* __restrict__ out, int n, int nb,
                                      long long units) {
    grid_launch_dependents();
    grid_wait_prior();
    constexpr int UPB = X16<6>::TB / 16;   // 210 units per tile-block
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        const long long tb = u / UPB;
        const int o = (int)(u - tb * UPB);
        const long long tile = tb / nb;
        const int b = (int)(tb - tile * nb);
        uint32_t v[4];
        for (int p = 0; p < 4; ++p) {
            // piece p of the unit: a row and a 4-byte offset inside its block
            int row, off;
            if (o < 16) {                      // scales of row o
                row = o;
                off = 192 + 4 * p;
            } else if (o < 18) {               // d of rows 8(o-16) + 2p, + 1
                row = -1;
                off = 0;
            } else if (o < 146) {              // ql pieces
                const int j = (o - 18) >> 5, L = (o - 18) & 31;
                row = (L >> 2) + (j >= 2 ? 8 : 0);
                off = 64 * (j & 1) + 16 * p + 4 * (L & 3);
            } else {                           // qh pieces, (h, s) = p >> 1, p & 1
                const int j = (o - 146) >> 5, L = (o - 146) & 31;
                row = (L >> 2) + 8 * j;
                off = 128 + 32 * (p >> 1) + 16 * (p & 1) + 4 * (L & 3);
            }
            uint32_t x = 0;
            if (row >= 0) {
                const long long r = tile * TR + row;
                if (r < n) {
                    const uint16_t* q = reinterpret_cast<const uint16_t*>(w + ((size_t)r * nb + b) * Q6K_BYTES + off);
                    x = (uint32_t)q[0] | ((uint32_t)q[1] << 16);
                }
            } else {
                for (int e = 0; e < 2; ++e) {
                    const long long r = tile * TR + 8 * (o - 16) + 2 * p + e;
                    if (r < n) {
                        const uint16_t dv = *reinterpret_cast<const uint16_t*>(w + ((size_t)r * nb + b) * Q6K_BYTES + 208);
                        x |= (uint32_t)dv << (16 * e);
                    }
                }
            }
            v[p] = x;
        }
        reinterpret_cast<uint4*>(out)[u] = make_uint4(v[0], v[1], v[2], v[3]);
    }
}

}  // namespace x16

size_t x16_bytes(int fmt, long long n, int k) {
    const int tb = fmt == 6 ? x16::X16<6>::TB : x16::X16<4>::TB;
    return (size_t)((n + x16::TR - 1) / x16::TR) * (k / QK) * tb;
}

cudaError_t launch_repack_x16(int fmt, const uint8_t* w, uint8_t* out, int n, int k, cudaStream_t stream) {
    const long long units = (long long)x16_bytes(fmt, n, k) / 16;
    long long grid = (units + 255) / 256;
    const long long cap = (long long)num_sms() * 8;
    if (grid > cap) grid = cap;
    if (fmt == 6)
        return launch_kernel(x16::repack_x16_q6K_kernel, dim3((unsigned)grid), dim3(256), 0, stream, w, out, n,
                             k / QK, units);
    return launch_kernel(x16::repack_x16_q4K_kernel, dim3((unsigned)grid), dim3(256), 0, stream, w, out, n, k / QK,
                         units);
}

template <int FMT>
static cudaError_t gemv_x16(const uint8_t* w, const uint8_t* xq, float* y, int m, int n, int k, cudaStream_t stream) {
    x16::Args A;
    A.w = w;
    A.xq = xq;
    A.y = y;
    A.fault = fault_word();
    if (!A.fault) return cudaErrorInvalidDevicePointer;
    A.m = m;
    A.n = n;
    A.nb = k / QK;
    A.ntiles = (n + x16::TR - 1) / x16::TR;
    int kl = 0;
    while (kl < 4 && (A.nb % (2 << kl)) == 0) ++kl;
    A.kw_log2 = kl;
    A.prefetch = overlap_mode() >= 2 ? 1 : 0;
    A.kmlo = 0x000F000Fu;
    A.kmhi = 0x00F000F0u;
    A.kmagic = 0x64006400u;
    A.k2p24 = 1u << 24;
    A.km1056 = 0xE420E420u;
    A.k0f = 0x0F0F0F0Fu;
    A.k30 = 0x30303030u;
    constexpr int SMEM = x16::smem_bytes<FMT>();
    cudaError_t e = cudaFuncSetAttribute(x16::gemv_x16_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    int grid = num_sms();
    if (grid > A.ntiles) grid = A.ntiles;
    return launch_kernel(x16::gemv_x16_kernel<FMT>, dim3((unsigned)grid), dim3(x16::THREADS), (size_t)SMEM, stream,
                         A);
}

cudaError_t launch_gemv_x16(int fmt, const uint8_t* w, const uint8_t* xq, float* y, int m, int n, int k,
                            cudaStream_t stream) {
    return fmt == 6 ? gemv_x16<6>(w, xq, y, m, n, k, stream) : gemv_x16<4>(w, xq, y, m, n, k, stream);
}

}  // namespace plm
