// Prefill GEMM over packed K-quant weights (q2_K .. q6_K) on the
// 5th-generation tensor cores (tcgen05, kind::f16), for m >= 9 activation rows
// (PocketLLM "What it runs": weights stay packed and are decoded inside the
// kernel; the matmul is a dense contraction once m is large).
//
// Exactness.  Per 256-weight block the method needs exact integers:
//   q4_K: isum = sum_j sc_j * sum_l q*q8 and msum = sum_g m_(g/2) * bsum_g,
//         term = d_x*d_w*isum - dmin_x*d_w*msum;
//   q5_K: as q4_K with 5-bit q (sc*q <= 63*31 = 1953, still exact in f16);
//   q2_K: as q4_K with 2-bit q and 16 (sc, m) pairs;
//   q3_K: isum over (s-32)*(q3+4), msum = sum_g 4 (s_g-32) bsum_g, dmin = d;
//   q6_K: isum = sum_g sc_g * sum_l (q6-32)*q8, term = d_x*d_w*isum.
// The operands are integer-valued and exact in f16: activation codes q8 in
// [-128, 127]; q4_K weights sc*q <= 945; bsums in [-2048, 2048]; mins <= 63.
// q6_K scales are int8, so sc*(q6-32) can reach 4096 and is not always exact
// in f16: the scale is split as sc = 16*hi + lo and the exact operands
// 16*hi*(q6-32) and lo*(q6-32) are contracted one after the other.  Products
// and partial sums are integers accumulated in f32, exact while below 2^24
// (only an adversarial block can exceed it; the f32 rounding there is far
// inside the 1e-4 tolerance).  Because d, dmin and d_x change every block,
// each block accumulates into fresh TMEM columns and is drained and scaled in
// f32.
//
// Tile: 128 weight rows (MMA M, TMEM lanes) x 128 activation rows (MMA N,
// TMEM columns).  gemm_tm_kernel (q2_K .. q5_K, and q6_K on shapes whose
// blocks come by TMA) keeps the decoded A operand in tensor memory; its roles
// are described above it.  gemm_kernel is the q6_K path for the other shapes:
//   producer warpgroup (warps 0-3): thread t reads weight row t's 210-byte
//     block one block ahead with its own loads and decodes it into the two
//     A operand tiles (f16, 128-byte swizzled K-major, one 64-wide K stage
//     at a time), writes the per-block scales, and thread 0 issues the TMA
//     load of the activation stage from the workspace the pre-pass fills;
//   the epilogue warpgroup (warps 4-7): drains D_hi and D_lo of each block
//     from TMEM, applies the scales and accumulates in registers; stores y;
//   warp 8 (one thread): issues the MMAs (M=128, N=128, K=16) and commits.
// A ring of 3 operand stages, double-buffered scales and double-buffered
// TMEM accumulators (2 x (128 + 128) columns) keep the roles overlapped.
// Every wait is bounded; a wait that runs out records a fault and the kernel
// winds down.
#include <cuda.h>
#include <cuda_fp16.h>

#include <cstring>
#include <type_traits>

#include "plm_device.cuh"
#include "plm_internal.h"

namespace plm {

constexpr int GT = 128;                 // tile rows (weights) and columns (activations)
constexpr int KS = 64;                  // K per operand stage (one 128-byte swizzle row)
constexpr int TILE_BYTES = GT * KS * 2; // 16 KB per operand tile
constexpr int XROW = 272;               // XIN: staged bytes per activation row and block
constexpr int XSTAGE_BYTES = GT * XROW; // XIN: one staging buffer of a block's codes
// Roles: PWG producer warpgroups (warpgroup h decodes stages [4h/PWG, 4(h+1)/PWG)
// of every block), one epilogue warpgroup, one MMA warp; PWG per format below.
// XIN (no workspace): NCV more warps after the MMA warp widen the activation
// codes into the B tiles (xin_issue, xin_convert) in place of the TMA.
template <int PWG> struct GemmRoles {
    static constexpr int EPI_WARP0 = 4 * PWG;      // first epilogue warp
    static constexpr int MMA_WARP = EPI_WARP0 + 4;
    static constexpr int NCV = 2;
    static constexpr int threads(bool xin) { return (MMA_WARP + 1 + (xin ? NCV : 0)) * 32; }
};
// per (activation row, 256-value block) in the workspace: the 16 bsums of
// the q8_K block as f16 pairs, its d as f32 bits, three zero words
constexpr int AUXB = 48;

// q4_K: one A tile per stage plus per-block min operands; q6_K: two A tiles
// per stage (the high and low parts of the scale), no min term.
// BSLOTS: slots of the TMA-fed ring of raw weight blocks (WROW bytes per
// weight row) and activation side data; 0 for q6_K.
// PWG: producer warpgroups (q6_K keeps one: its rows are read per thread,
// whole, and need the registers).
// WPITCH: bytes per weight row in a block slot, the TMA box width (q2_K,
// q3_K: a 16-byte-aligned window around the block, an odd number of 16-byte
// units so that the producers' 16-byte reads of 32 rows hit distinct banks).
template <int FMT> struct GemmCfg;
template <> struct GemmCfg<2> {   // q2_K: 84-byte blocks, window of 96 bytes at most
    static constexpr int ATILES = 1, NSTAGE = 4, MINB = 2 * TILE_BYTES, BSLOTS = 2, WROW = Q2K_BYTES, PWG = 2;
    static constexpr int WPITCH = 112;
};
template <> struct GemmCfg<3> {   // q3_K: 110-byte blocks, window of 124 bytes at most
    static constexpr int ATILES = 1, NSTAGE = 4, MINB = 2 * TILE_BYTES, BSLOTS = 2, WROW = Q3K_BYTES, PWG = 2;
    static constexpr int WPITCH = 144;
};
template <> struct GemmCfg<4> {
    static constexpr int ATILES = 1, NSTAGE = 4, MINB = 2 * TILE_BYTES, BSLOTS = 2, WROW = Q4K_BYTES, PWG = 2;
    static constexpr int WPITCH = WROW;
};
template <> struct GemmCfg<5> {   // q5_K: q4_K's operands, a fifth bit per weight
    static constexpr int ATILES = 1, NSTAGE = 4, MINB = 2 * TILE_BYTES, BSLOTS = 2, WROW = Q5K_BYTES, PWG = 2;
    static constexpr int WPITCH = WROW;
};
template <> struct GemmCfg<6> {
    static constexpr int ATILES = 2, NSTAGE = 3, MINB = 0, BSLOTS = 0, WROW = 0, PWG = 1;
    static constexpr int WPITCH = 0;
};
// q6_K in the tensor-memory kernel (gemm_tm_kernel<Q6TM>): 210-byte blocks
// in 16-byte windows of at most 224 bytes, 15 units a row
constexpr int Q6TM = 7;
template <> struct GemmCfg<Q6TM> {
    static constexpr int ATILES = 1, NSTAGE = 4, MINB = 0, BSLOTS = 2, WROW = Q6K_BYTES, PWG = 2;
    static constexpr int WPITCH = 240;
};

template <int FMT, bool XIN>
struct GemmSmem {
    // offsets from the 1024-aligned base
    static constexpr int NSTAGE = GemmCfg<FMT>::NSTAGE;
    static constexpr int STAGE = (GemmCfg<FMT>::ATILES + 1) * TILE_BYTES;   // A tile(s), then B
    static constexpr int RING = 0;
    static constexpr int MIN = RING + NSTAGE * STAGE;                        // q4_K: 2 x 16 KB
    static constexpr int SCL = MIN + GemmCfg<FMT>::MINB;                     // 2 x (d, dmin, dx) x 128 f32
    static constexpr int WT = GT * GemmCfg<FMT>::WROW;                       // raw weight tile of one block
    static constexpr int BTX = WT + GT * AUXB;                               // bytes landing per block slot
    static constexpr int BSLOT = (BTX + 1023) & ~1023;
    static constexpr int BRING = (SCL + 2 * 3 * GT * 4 + 1023) & ~1023;
    static constexpr int XST = BRING + GemmCfg<FMT>::BSLOTS * BSLOT;        // XIN: 2 staging buffers
    static constexpr int BAR = XST + (XIN ? 2 * XSTAGE_BYTES : 0);
    static constexpr int NBAR = 2 * NSTAGE + 8 + 2 * GemmCfg<FMT>::BSLOTS + (XIN ? 4 : 0);
    static constexpr int TMEMP = BAR + NBAR * 8;
    static constexpr int BYTES = TMEMP + 16;
    static constexpr int ALLOC = BYTES + 1024;   // + alignment slack
    static_assert(ALLOC <= 227 * 1024, "shared memory");
};

// byte offset of element (row, k) in a 128-row x 64-wide f16 tile with the
// 128-byte swizzle (16-byte chunk index XOR row % 8)
__device__ __forceinline__ uint32_t sw128_chunk(int row, int chunk) {
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + (((chunk ^ (row & 7)) & 7) << 4));
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle,
// 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor: D f32, A/B f16, both K-major, M = 128, N = 128
constexpr uint32_t IDESC_F16_128x128 = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t da, uint64_t db, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(dtmem), "l"(da), "l"(db), "r"(IDESC_F16_128x128), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// thread-block cluster: barrier over all threads of all its CTAs, rank, peer shared memory
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float4 ld_peer_f4(const void* local, uint32_t rank) {
    uint32_t addr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(local)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[8]) { tmem_ld8(taddr, r); }
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
                 "%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Two f32 values in one 64-bit register and the packed f32x2 arithmetic on
// them (each half rounded as its scalar instruction would round it)
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---------------------------------------------------------------------------
// In-kernel activation operand (the entry points without a workspace).
// Converter warps widen the q8_K codes of the tile's 128 activation rows into
// the f16 B tiles, in the layout the TMA would write.  Converter warp 0 brings
// each block's codes into shared memory a block ahead of use: per activation
// row one bulk copy of XROW bytes starting at the 16-byte boundary at or below
// the row's 256 codes (the window ends inside the row's q8_K block and starts
// no lower than the 16-byte chunk holding xq's first byte), into one of two
// staging buffers.  All converter threads then widen the block's stages from
// there: a code q becomes f16 (1024 + (q + 128)) - 1152 = q, exact; rows past
// m become zeros.  The per-block side data (bsums as f16 pairs, d) is loaded
// a block ahead into registers and written where the TMA would put it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}


// Converter warp 0: block blk's codes of activation rows i0 .. into a
// staging buffer.  xmap (when xq is 16-byte aligned and a row of q8_K blocks
// a multiple of 16 bytes, i.e. nb % 4 == 0): one TMA box of 128 rows x 68
// four-byte words from the 16-byte boundary at or below the block's codes
// (the same for every row; rows past m arrive as zeros).  Otherwise one bulk
// copy per row.
__device__ __forceinline__ void xin_issue(uint8_t* st, uint64_t* bar, const CUtensorMap* xmap, bool xtma,
                                          const uint8_t* xq, int nb, int m, int i0, int blk, int lane) {
    if (xtma) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, (uint32_t)XSTAGE_BYTES);
            tma_load_2d(st, xmap, (((Q8K_BYTES * blk + 4) & ~15) >> 2), i0, bar);
        }
        return;
    }
    const int valid = min(GT, m - i0);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(valid * XROW));
    __syncwarp();
    for (int r = lane; r < valid; r += 32) {
        const uint8_t* src = xq + ((size_t)(i0 + r) * nb + blk) * Q8K_BYTES + 4;
        bulk_g2s(st + r * XROW, src - ((uintptr_t)src & 15u), XROW, bar);
    }
}

// The widening work of a staged block is 512 units: unit k is stage c = k /
// 128 and, within it, row phase ph = (k % 128) / 16 and word wi = k % 16,
// i.e. the four codes 64c + 4wi .. of the 16 rows ph, ph + 8, ..., ph + 120.
// Rows eight apart share their swizzle pattern and, since 8 * 292 * nb is a
// multiple of 16, their skew in the staging window, so every load and store
// of a unit sits at a constant offset from the first.
__device__ __forceinline__ void xin_unit(const uint8_t* st, uint8_t* tile, uint32_t sk, int c, int ph, int wi) {
    const uint8_t* src = st + ph * XROW + sk + c * KS + 4 * wi;
    uint8_t* dst = tile + ph * 128 + ((((wi >> 1) ^ ph) & 7) << 4) + 8 * (wi & 1);
    const __half2 off = bits_h2(0x64806480u);   // 1152, 1152
    uint32_t v[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) v[t] = *reinterpret_cast<const uint32_t*>(src + t * 8 * XROW);
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        const uint32_t x = v[t] ^ 0x80808080u;   // q + 128 per byte
        const uint32_t lo = h2_bits(__hsub2(bits_h2(prmt(x, 0x64646464u, 0x4140u)), off));
        const uint32_t hi = h2_bits(__hsub2(bits_h2(prmt(x, 0x64646464u, 0x4342u)), off));
        *reinterpret_cast<uint2*>(dst + t * 1024) = make_uint2(lo, hi);   // rows 8 apart: 1 KB apart
    }
}

// The skew of the rows of phase ph in their staging windows: the codes'
// address mod 16 (a 32-bit wrap keeps it).
__device__ __forceinline__ uint32_t xin_skew(const uint8_t* xq, int nb, int i0, int blk, int ph) {
    return ((uint32_t)(uintptr_t)xq + 4u + (uint32_t)Q8K_BYTES * (uint32_t)blk +
            (uint32_t)Q8K_BYTES * (uint32_t)nb * (uint32_t)(i0 + ph)) & 15u;
}

// One staged block: converter thread u (of NT, a multiple of 32) takes units
// u, u + NT, ... in order, so each warp meets the stages in order and has
// units in every stage.  Before its first unit of stage c it waits for the
// slot (wait_slot(c)); after its last it publishes the stage (done(c)).
template <int NT, class WaitSlot, class Tile, class Done>
__device__ __forceinline__ bool xin_block(const uint8_t* st, const uint8_t* xq, int nb, int i0, int blk, int u,
                                          WaitSlot wait_slot, Tile tile, Done done) {
    // warp-uniform stages, and every warp meets every stage (steps of at most 128 units)
    static_assert(NT % 32 == 0 && NT <= 128, "converter threads");
    constexpr int PER = (512 + NT - 1) / NT;
    const int k0 = u & ~31;   // the warp's first unit
    int cur = -1;
#pragma unroll 1
    for (int t = 0; t < PER; ++t) {   // not unrolled: the kernel's roles share the instruction cache
        const int kw = k0 + NT * t;   // warp-uniform
        if (kw >= 512) break;
        const int k = u + NT * t;
        const int c = kw >> 7;
        if (c != cur) {
            if (cur >= 0) done(cur);
            if (!wait_slot(c)) return false;
            cur = c;
        }
        const int ph = (k >> 4) & 7, wi = k & 15;
        xin_unit(st, tile(c), xin_skew(xq, nb, i0, blk, ph), c, ph, wi);
    }
    done(cur);
    return true;
}

// Per-row copies leave the staging rows past m untouched: zero them once
// (both buffers) so that those rows widen to zeros.
__device__ __forceinline__ void xin_zero_tail(uint8_t* xst, int valid, int u, int nt) {
    for (int o = valid * XROW / 16 + u; o < GT * XROW / 16; o += nt) {
        reinterpret_cast<uint4*>(xst)[o] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(xst + XSTAGE_BYTES)[o] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Side data of one block for the tile's rows u, u + NT, ...: the eight words
// of bsums and d, loaded a block ahead, then written as AUXB bytes per row
// (the 16 bsums as f16 pairs, |bsum| <= 2048: exact; d; three zero words).
template <int NT>
struct XinSide {
    static constexpr int ROWS = (GT + NT - 1) / NT;
    uint32_t v[ROWS][9];
};

template <int NT>
__device__ __forceinline__ void xin_side_load(XinSide<NT>& S, const uint8_t* xq, int nb, int m, int i0, int blk,
                                              int u) {
#pragma unroll
    for (int r = 0; r < XinSide<NT>::ROWS; ++r) {
        const int t = u + NT * r, i = i0 + t;
        const bool valid = t < GT && i < m;
        const uint8_t* b = xq + ((size_t)(valid ? i : 0) * nb + blk) * Q8K_BYTES;
#pragma unroll
        for (int g = 0; g < 8; ++g)
            S.v[r][g] = valid ? __ldg(reinterpret_cast<const uint32_t*>(b + 4 + QK) + g) : 0u;
        S.v[r][8] = valid ? __ldg(reinterpret_cast<const uint32_t*>(b)) : 0u;
    }
}

template <int NT>
__device__ __forceinline__ void xin_side_store(const XinSide<NT>& S, uint8_t* side, int u) {
#pragma unroll
    for (int r = 0; r < XinSide<NT>::ROWS; ++r) {
        const int t = u + NT * r;
        if (t >= GT) break;
        uint32_t o[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const uint32_t v = S.v[r][g];
            o[g] = h2_bits(__halves2half2(__int2half_rn((int)(int16_t)(v & 0xFFFFu)),
                                          __int2half_rn((int)(int16_t)(v >> 16))));
        }
        uint4* dst = reinterpret_cast<uint4*>(side + t * AUXB);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        dst[2] = make_uint4(S.v[r][8], 0u, 0u, 0u);
    }
}

// SwiGLU of a gate/up pair: silu(g) * u = g / (1 + e^-g) * u
__device__ __forceinline__ float swiglu1(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}


// One producer warpgroup's share of a q4_K / q5_K row (tensor-memory GEMM):
// the header and the qs (q5_K: and qh) of its two chunks 2h, 2h + 1 with
// their f16x2 constants, so a warpgroup holds half the block in registers.
template <int FMT>
struct QxKHalf {
    uint4 hdr;
    uint4 qs[4];      // chunk 2h: qs[0..1], chunk 2h + 1: qs[2..3]
    uint4 qh[2];      // q5_K: the fifth bits of all 256 weights
    float d, dmin;
    uint32_t sc_lo2[2], off_lo2[2], sc_hi2[2], off_hi2[2];
};

template <int FMT>
__device__ __forceinline__ void qxK_half_load(QxKHalf<FMT>& R, const uint8_t* row, int half) {
    const uint4* p = reinterpret_cast<const uint4*>(row);
    constexpr int QW = FMT == 5 ? 3 : 1;   // first qs word (q5_K: after qh[32])
    R.hdr = p[0];
    if constexpr (FMT == 5) {
        R.qh[0] = p[1];
        R.qh[1] = p[2];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) R.qs[u] = p[QW + 4 * half + u];
}

// d, dmin and the multiply-add constants of chunks 2h, 2h + 1: the 6-bit s as f16
// through the 1024 + s bit pattern; low nibbles (1024 + q) * sc - 1024 * sc,
// high nibbles in place (1024 + 16 q) * sc / 16 - 64 * sc, all exact
template <int FMT>
__device__ __forceinline__ void qxK_half_prepare(QxKHalf<FMT>& R, int half) {
    const uint4 hdr = R.hdr;
    R.d = half_bits_to_float(hdr.x);
    R.dmin = half_bits_to_float(hdr.x >> 16);
    const uint32_t scw = half ? ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u)) : (hdr.y & 0x3F3F3F3Fu);
#pragma unroll
    for (int cl = 0; cl < 2; ++cl) {
        const uint32_t slo = (scw >> (16 * cl)) & 0xFFu, shi = (scw >> (16 * cl + 8)) & 0xFFu;
        const __half2 lo2 = __hsub2(bits_h2(0x64006400u | slo | (slo << 16)), bits_h2(0x64006400u));
        const __half2 hi2 = __hsub2(bits_h2(0x64006400u | shi | (shi << 16)), bits_h2(0x64006400u));
        R.sc_lo2[cl] = h2_bits(lo2);
        R.off_lo2[cl] = h2_bits(__hmul2(lo2, bits_h2(0xE400E400u)));   // x (-1024)
        R.sc_hi2[cl] = h2_bits(__hmul2(hi2, bits_h2(0x2C002C00u)));    // x 1/16
        R.off_hi2[cl] = h2_bits(__hmul2(hi2, bits_h2(0xD400D400u)));   // x (-64)
    }
}

// the min operand's first 16 K positions: m_(g/2) for K g (f16 pairs)
__device__ __forceinline__ void qxK_min_pairs(const uint4 hdr, uint32_t (&mv)[8]) {
    const uint32_t m_a = hdr.z & 0x3F3F3F3Fu;
    const uint32_t m_b = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const uint32_t mm = ((g < 4 ? m_a : m_b) >> (8 * (g & 3))) & 0xFFu;
        mv[g] = h2_bits(__hsub2(bits_h2(0x64006400u | mm | (mm << 16)), bits_h2(0x64006400u)));
    }
}

// chunk c = 2h + CL (weights 64c .. 64c + 63) into the 32 tensor-memory columns of
// the row: column i holds K positions 2i, 2i + 1 as an f16 pair; K 0..31 are the low
// nibbles of qs[32c .. 32c + 31] times sc_(2c), K 32..63 the high nibbles times
// sc_(2c+1) (q5_K: the fifth bit from qh[l], bit 2c resp. 2c + 1)
template <int FMT, int CL>
__device__ __forceinline__ void qxK_half_stage_regs(const QxKHalf<FMT>& R, int c, uint32_t (&v)[32]) {
    const uint4 qa = R.qs[2 * CL], qb = R.qs[2 * CL + 1];
    const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const __half2 slo = bits_h2(R.sc_lo2[CL]), olo = bits_h2(R.off_lo2[CL]);
    const __half2 shi = bits_h2(R.sc_hi2[CL]), ohi = bits_h2(R.off_hi2[CL]);
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t w = q[2 * ch + h];
            const uint32_t x01 = __byte_perm(w, 0, 0x4140), x23 = __byte_perm(w, 0, 0x4342);
            uint32_t l01 = x01 & 0x000F000Fu, l23 = x23 & 0x000F000Fu;
            uint32_t u01 = x01 & 0x00F000F0u, u23 = x23 & 0x00F000F0u;
            if constexpr (FMT == 5) {
                const uint4 qhv = R.qh[ch >> 1];
                const uint32_t qw[4] = {qhv.x, qhv.y, qhv.z, qhv.w};
                const uint32_t b = qw[2 * (ch & 1) + h];
                const uint32_t h01 = __byte_perm(b, 0, 0x4140), h23 = __byte_perm(b, 0, 0x4342);
                l01 |= ((h01 >> (2 * c)) & 0x00010001u) << 4;
                l23 |= ((h23 >> (2 * c)) & 0x00010001u) << 4;
                u01 |= ((h01 >> (2 * c + 1)) & 0x00010001u) << 8;
                u23 |= ((h23 >> (2 * c + 1)) & 0x00010001u) << 8;
            }
            v[4 * ch + 2 * h] = h2_bits(__hfma2(bits_h2(l01 | 0x64006400u), slo, olo));
            v[4 * ch + 2 * h + 1] = h2_bits(__hfma2(bits_h2(l23 | 0x64006400u), slo, olo));
            v[16 + 4 * ch + 2 * h] = h2_bits(__hfma2(bits_h2(u01 | 0x64006400u), shi, ohi));
            v[16 + 4 * ch + 2 * h + 1] = h2_bits(__hfma2(bits_h2(u23 | 0x64006400u), shi, ohi));
        }
    }
}


// f16 pair of two small non-negative integers a, b < 1024 (exact)
__device__ __forceinline__ __half2 small_pair(uint32_t a, uint32_t b) {
    return __hsub2(bits_h2(0x64006400u | a | (b << 16)), bits_h2(0x64006400u));
}

// One producer warpgroup's share of a q2_K / q3_K row: the qs words of its
// half h (bytes 32h .. 32h + 31), the scale words (all of them: the min
// operand needs every group's), q3_K's hmask, and the d word.  Each range is
// read as whole 16-byte units of the window (at a runtime offset) and
// shifted down by the tile-uniform skew sk.
template <int FMT>
struct QlowHalf {
    uint32_t qs[8];
    uint32_t sc[4];   // q2_K: scale bytes 0..15; q3_K: words 24..26 (sc[3] unused)
    uint32_t hm[8];   // q3_K: hmask[32]
    float d, dmin;
};

// words [first, first + N) of the block: window units from first / 4 on
// (first a multiple of 4), then down by sk bytes
template <int N>
__device__ __forceinline__ void qlow_words(const uint8_t* row, int first, int sk, uint32_t (&out)[N]) {
    constexpr int U = (N + 4 + 3) / 4;   // units covering N + 1 words past a shift of up to 3 words
    uint32_t x[4 * U];
    const uint4* p = reinterpret_cast<const uint4*>(row) + (first >> 2);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint4 q = p[u];
        x[4 * u] = q.x; x[4 * u + 1] = q.y; x[4 * u + 2] = q.z; x[4 * u + 3] = q.w;
    }
    const uint32_t sh = (uint32_t)(sk & 2) * 8u;   // 0 or 16 bits
    switch (sk >> 2) {
        case 0:
#pragma unroll
            for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(x[i], x[i + 1], sh);
            break;
        case 1:
#pragma unroll
            for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(x[i + 1], x[i + 2], sh);
            break;
        case 2:
#pragma unroll
            for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(x[i + 2], x[i + 3], sh);
            break;
        default:
#pragma unroll
            for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(x[i + 3], x[i + 4], sh);
            break;
    }
}

template <int FMT>
__device__ __forceinline__ void qlow_half_load(QlowHalf<FMT>& R, const uint8_t* row, int sk, int half) {
    if constexpr (FMT == 2) {
        qlow_words<8>(row, 4 + 8 * half, sk, R.qs);
        qlow_words<4>(row, 0, sk, R.sc);
        uint32_t dw[1];
        qlow_words<1>(row, 20, sk, dw);
        R.d = half_bits_to_float(dw[0] & 0xFFFFu);    // bytes 80, 81
        R.dmin = half_bits_to_float(dw[0] >> 16);     // bytes 82, 83
    } else {
        qlow_words<8>(row, 8 + 8 * half, sk, R.qs);
        qlow_words<8>(row, 0, sk, R.hm);
        uint32_t sw[4];
        qlow_words<4>(row, 24, sk, sw);               // scales (words 24..26), d (word 27)
        R.sc[0] = sw[0]; R.sc[1] = sw[1]; R.sc[2] = sw[2]; R.sc[3] = 0;
        R.d = half_bits_to_float(sw[3] & 0xFFFFu);    // bytes 108, 109
        R.dmin = R.d;                                 // the -4 S bsum part
    }
}

// q3_K six-bit scale of group g = 8 gh + gl (gl = g % 8 known at compile time)
__device__ __forceinline__ uint32_t q3K_s6h(const uint32_t (&sc)[4], int gl, int gh) {
    const int g4 = gl & 3;
    const uint32_t lo = (sc[gl >> 2] >> (8 * g4 + 4 * gh)) & 15u;
    const uint32_t hi = (sc[2] >> (8 * g4 + 2 * (2 * gh + (gl >> 2)))) & 3u;
    return lo | (hi << 4);
}

template <int FMT>
__device__ __forceinline__ void qlow_half_min_pairs(const QlowHalf<FMT>& R, uint32_t (&mv)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {   // groups 2i, 2i + 1
        if constexpr (FMT == 2) {
            const uint32_t w = R.sc[i >> 1] >> (16 * (i & 1));
            mv[i] = h2_bits(small_pair((w >> 4) & 15u, (w >> 12) & 15u));
        } else {   // 4 S = 4 s6 - 128, exact
            const int g0 = 2 * i, g1 = 2 * i + 1;
            const __half2 sp = small_pair(q3K_s6h(R.sc, g0 & 7, g0 >> 3), q3K_s6h(R.sc, g1 & 7, g1 >> 3));
            mv[i] = h2_bits(__hfma2(sp, bits_h2(0x44004400u), bits_h2(0xD800D800u)));
        }
    }
}

// One producer warpgroup's share of a q6_K row (tensor-memory GEMM): half
// h = stages 2h, 2h + 1 = weights 128h .. 128h + 127, whose low four bits are
// ql[64h .. 64h + 63] and top two bits qh[32h .. 32h + 31]; the int8 scales
// and d.  Stage c = 2h + CL, K position p (0..63): code = (ql[64h + p] >> 4 CL
// & 15) | (qh[32h + p % 32] >> (4 CL + 2 (p >= 32)) & 3) << 4, group 4c + p / 16.
// Each scale is split as sc = 16 hi + lo (lo in 0..15): the two operands
// 16 hi (q - 32) (a multiple of 16 up to 4096 in magnitude) and lo (q - 32)
// are exact in f16 and go into the same accumulator.
struct Q6Half {
    uint32_t ql[16];
    uint32_t qh[8];
    uint32_t sc[4];   // the 16 int8 scales
    float d;
};

__device__ __forceinline__ void q6_half_load(Q6Half& R, const uint8_t* row, int sk, int half) {
    qlow_words<16>(row, 16 * half, sk, R.ql);
    qlow_words<8>(row, 32 + 8 * half, sk, R.qh);
    qlow_words<4>(row, 48, sk, R.sc);
    uint32_t dw[1];
    qlow_words<1>(row, 52, sk, dw);
    R.d = half_bits_to_float(dw[0] & 0xFFFFu);   // bytes 208, 209
}

// columns 16 P .. 16 P + 15 of stage c = 2h + CL (K positions 32 P .. 32 P + 31)
// of both operands
template <int CL, int P>
__device__ __forceinline__ void q6_half_stage_regs(const Q6Half& R, int h, uint32_t (&vh)[16], uint32_t (&vl)[16]) {
    const __half2 m1056 = bits_h2(0xE420E420u);   // -1056
#pragma unroll
    for (int gq = 0; gq < 2; ++gq) {              // the two 16-weight groups of these positions
        const int gl = 4 * CL + 2 * P + gq;       // group within the half
        const uint32_t w = h ? R.sc[2 + (gl >> 2)] : R.sc[gl >> 2];
        const int sc = (int)(int8_t)((w >> (8 * (gl & 3))) & 0xFFu);
        const __half2 hi16 = __float2half2_rn((float)((sc >> 4) * 16));
        const uint32_t lo = (uint32_t)(sc & 15);
        const __half2 lo2 = small_pair(lo, lo);
        const __half2 lo_off = __hmul2(lo2, m1056);   // -1056 lo, exact
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int wi = 8 * P + 4 * gq + u;         // positions 4 wi .. 4 wi + 3
            const uint32_t nib = (R.ql[wi] >> (4 * CL)) & 0x0F0F0F0Fu;
            const uint32_t hb = (R.qh[wi & 7] >> (4 * CL + 2 * (wi >> 3))) & 0x03030303u;
            const uint32_t code = nib | (hb << 4);
            const __half2 x01 = bits_h2(prmt(code, 0x64646464u, 0x4140u));   // 1024 + q
            const __half2 x23 = bits_h2(prmt(code, 0x64646464u, 0x4342u));
            const int col = 8 * gq + 2 * u;
            vh[col] = h2_bits(__hmul2(__hadd2(x01, m1056), hi16));
            vh[col + 1] = h2_bits(__hmul2(__hadd2(x23, m1056), hi16));
            vl[col] = h2_bits(__hfma2(x01, lo2, lo_off));
            vl[col + 1] = h2_bits(__hfma2(x23, lo2, lo_off));
        }
    }
}

// f16 of 4^-j and of -1024 * 4^-j
__device__ __forceinline__ uint32_t pow4_inv_bits(int j) { return 0x3C00u - 0x0800u * (uint32_t)j; }
__device__ __forceinline__ uint32_t neg1024_pow4_inv_bits(int j) { return 0xE400u - 0x0800u * (uint32_t)j; }

template <int FMT, int CL>
__device__ __forceinline__ void qlow_half_stage_regs(const QlowHalf<FMT>& R, int h, uint32_t (&v)[32]) {
    constexpr int j0 = 2 * CL;   // stage c = 2h + CL: groups 8h + 4 CL + gg
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) {
        const int gl = 4 * CL + gg;   // group within the half
        const int j = j0 + (gg >> 1), p = gg & 1;
        // the group's multiply-add constants
        __half2 sg;
        if constexpr (FMT == 2) {
            const uint32_t w = h ? R.sc[2 + (gl >> 2)] : R.sc[gl >> 2];   // scale bytes of groups 8h ..
            const uint32_t sc = (w >> (8 * (gl & 3))) & 15u;
            sg = small_pair(sc, sc);
        } else {
            const uint32_t s6 = q3K_s6h(R.sc, gl, h);
            sg = __hsub2(bits_h2(0x64006400u | s6 | (s6 << 16)), bits_h2(0x64206420u));   // s6 - 32
        }
        const uint32_t m1 = pow4_inv_bits(j), m2 = neg1024_pow4_inv_bits(j);
        const __half2 mul = __hmul2(sg, bits_h2(m1 | (m1 << 16)));
        const __half2 add = __hmul2(sg, bits_h2(m2 | (m2 << 16)));
        const uint32_t qmask = 0x00030003u << (2 * j);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t qw = R.qs[4 * p + u];   // qs[32h + 16p + 4u ..]
            uint32_t x01 = __byte_perm(qw, 0, 0x4140) & qmask, x23 = __byte_perm(qw, 0, 0x4342) & qmask;
            if constexpr (FMT == 3) {
                const uint32_t hw = R.hm[4 * p + u];   // hmask bytes 16p + 4u ..
                const uint32_t h01 = __byte_perm(hw, 0, 0x4140), h23 = __byte_perm(hw, 0, 0x4342);
                // hbit (bit 4h + j of the byte) to bit 2j + 2 of each half: up by j + 2, down by 4h
                const uint32_t hmask = 0x00010001u << (2 * j + 2);
                x01 |= ((h01 << (j + 2)) >> (4 * h)) & hmask;
                x23 |= ((h23 << (j + 2)) >> (4 * h)) & hmask;
            }
            v[8 * gg + 2 * u] = h2_bits(__hfma2(bits_h2(x01 | 0x64006400u), mul, add));
            v[8 * gg + 2 * u + 1] = h2_bits(__hfma2(bits_h2(x23 | 0x64006400u), mul, add));
        }
    }
}

// q6_K: stage c (weights 64c .. 64c+63) lies in half h = c/2, quarters
// 2(c&1) and 2(c&1)+1.  K position p < 32 is weight 128h + 32*2(c&1) + p,
// p >= 32 is weight 128h + 32*(2(c&1)+1) + p - 32; their low four bits come
// from ql[64h + p] (resp. ql[64h + 32 + p - 32]) -- low nibble for c even,
// high nibble for c odd -- and their top two bits from qh[32h + (p mod 32)]
// (bits 4(c&1) .. +1 for p < 32, 4(c&1)+2 .. +3 otherwise).  Position p
// belongs to the 16-group 4c + p/16.  Each int8 scale is split as
// sc = 16*hi + lo (lo in 0..15), so that both operand tiles hi*(q6-32) and
// lo*(q6-32) are exact in f16 for every int8 scale.
struct Q6KRow {
    uint32_t raw[53];        // the 210-byte block, word i = bytes 4i .. 4i+3 (word 52: bytes 208, 209)
    float d;
};

__device__ __forceinline__ void q6K_row_load(Q6KRow& R, const uint8_t* blk, bool valid) {
    if (!valid) {
#pragma unroll
        for (int i = 0; i < 53; ++i) R.raw[i] = 0;
        return;
    }
    // the block starts 2-byte aligned; read aligned words and realign
    const uintptr_t addr = reinterpret_cast<uintptr_t>(blk);
    const int mis = (int)(addr & 3);                    // 0 or 2
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(addr - mis);
#pragma unroll
    for (int i = 0; i < 52; ++i) R.raw[i] = __ldg(aw + i);
    // word 52: with mis == 2 the aligned word at 208 ends at the block's last
    // byte; with mis == 0 only the last two bytes exist
    const uint32_t last = mis ? __ldg(aw + 52) : (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(blk + 208));
    if (mis) {
#pragma unroll
        for (int i = 0; i < 51; ++i) R.raw[i] = __funnelshift_r(R.raw[i], R.raw[i + 1], 16);
        R.raw[51] = __funnelshift_r(R.raw[51], last, 16);
        R.raw[52] = last >> 16;
    } else {
        R.raw[52] = last;
    }
}

// writes stage c of the row as two f16 tiles: hi*(q6-32) and lo*(q6-32)
__device__ __forceinline__ void q6K_row_stage(const Q6KRow& R, int c, uint8_t* tile_hi, uint8_t* tile_lo,
                                              int row) {
    const int h = c >> 1, part = c & 1;
    const uint32_t scw = R.raw[48 + c];                  // scales 4c .. 4c+3
    __half2 shi[4], ohi[4], slo[4], olo[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int sc = (int)(int8_t)((scw >> (8 * g)) & 0xFF);
        const float hi = (float)(sc >> 4), lo = (float)(sc & 15);
        // (1024 + q6) * s - 1056 * s = (q6 - 32) * s, exact
        shi[g] = __float2half2_rn(hi);
        ohi[g] = __float2half2_rn(-1056.0f * hi);
        slo[g] = __float2half2_rn(lo);
        olo[g] = __float2half2_rn(-1056.0f * lo);
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {                      // positions 8ch .. 8ch+7
        const int second = ch >> 2;                       // 0: p < 32, 1: p >= 32
        const int g = ch >> 1;                            // 16-group within the stage
        uint32_t vh[4], vl[4];
#pragma unroll
        for (int wv = 0; wv < 2; ++wv) {
            const int u = 2 * (ch & 3) + wv;              // word index: positions 4u .. 4u+3 of the half
            const uint32_t ql = R.raw[16 * h + 8 * second + u];
            const uint32_t qh = R.raw[32 + 8 * h + u];
            const uint32_t nib = part ? ((ql >> 4) & 0x0F0F0F0Fu) : (ql & 0x0F0F0F0Fu);
            const uint32_t hb = (qh >> (4 * part + 2 * second)) & 0x03030303u;
            const uint32_t code = nib | (hb << 4);
            const uint32_t x01 = (__byte_perm(code, 0, 0x4140) & 0x003F003Fu) | 0x64006400u;
            const uint32_t x23 = (__byte_perm(code, 0, 0x4342) & 0x003F003Fu) | 0x64006400u;
            vh[2 * wv] = h2_bits(__hfma2(bits_h2(x01), shi[g], ohi[g]));
            vh[2 * wv + 1] = h2_bits(__hfma2(bits_h2(x23), shi[g], ohi[g]));
            vl[2 * wv] = h2_bits(__hfma2(bits_h2(x01), slo[g], olo[g]));
            vl[2 * wv + 1] = h2_bits(__hfma2(bits_h2(x23), slo[g], olo[g]));
        }
        *reinterpret_cast<uint4*>(tile_hi + sw128_chunk(row, ch)) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
        *reinterpret_cast<uint4*>(tile_lo + sw128_chunk(row, ch)) = make_uint4(vl[0], vl[1], vl[2], vl[3]);
    }
}

// ---------------------------------------------------------------------------
// The GEMM kernel
// ---------------------------------------------------------------------------
struct GemmArgs {
    const uint8_t* w;        // q2_K .. q6_K blocks [n][nb]
    const uint8_t* xq;       // q8_K [m][nb]
    float* y;                // [m][n]
    float* part;             // split K: partial sums [gridDim.z][m][n] (null: write y)
    const float* gate;       // GATE kernels (unsplit q4_K): y = silu(gate) * result, gate may be y itself
    int xtma;                // XIN: the staged codes come by TMA (xmap), else by one bulk copy per row
    int csplit;              // > 1: the grid's z CTAs of a tile form a cluster, rank 0 adds their partials
    unsigned* fault;
    int m, n, nb;
    int bsplit;              // blocks of K per split (blockIdx.z)
    int ty0;                 // the launch's first weight tile (grid y counts from it)
};

template <int FMT, bool XIN>
__global__ void __launch_bounds__(GemmRoles<GemmCfg<FMT>::PWG>::threads(XIN), 1) gemm_kernel(const __grid_constant__ CUtensorMap xmap,
                                                               const __grid_constant__ CUtensorMap wmap,
                                                               const __grid_constant__ CUtensorMap amap,
                                                               const GemmArgs A) {
    using L = GemmSmem<FMT, XIN>;
    constexpr int NSTAGE = L::NSTAGE;
    constexpr int PWG = GemmCfg<FMT>::PWG;
    constexpr int EPI_WARP0 = GemmRoles<PWG>::EPI_WARP0, MMA_WARP = GemmRoles<PWG>::MMA_WARP;
    constexpr int BOFF = GemmCfg<FMT>::ATILES * TILE_BYTES;   // B tile offset inside a stage
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint64_t* full = bars;                  // [NSTAGE], 4 arrivals (the stage's warpgroup) + TMA bytes (XIN: NCV arrivals)
    uint64_t* empty = bars + NSTAGE;        // [NSTAGE], MMA commit
    uint64_t* minfull = bars + 2 * NSTAGE;  // [2], one arrival per producer warp (min operands, scales)
    uint64_t* minempty = minfull + 2;       // [2], MMA commit
    uint64_t* tfull = minfull + 4;          // [2], MMA commit
    uint64_t* tempty = minfull + 6;         // [2], 4 epilogue-warp arrivals
    uint64_t* bfull = minfull + 8;          // [BSLOTS], TMA bytes of a weight block and its side data
    uint64_t* bempty = bfull + GemmCfg<FMT>::BSLOTS;   // [BSLOTS], one arrival per producer warp
    uint64_t* xfull = bempty + GemmCfg<FMT>::BSLOTS;   // XIN [2]: bulk-copy bytes of a staged block of codes
    uint64_t* xempty = xfull + 2;                      // XIN [2]: converter-warp arrivals once it is widened
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::TMEMP);
    float* scl = reinterpret_cast<float*>(sm + L::SCL);   // [2][3][128]: d, dmin, dx

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // x: activation tile, y: weight tile, so the CTAs that share a weight tile
    // run next to each other and its re-reads come from L2
    const int r0 = (blockIdx.y + A.ty0) * GT, i0 = blockIdx.x * GT;
    const int nb = A.nb;
    // this CTA's share of K: blocks [kb0, kb0 + kcount); loop indices below count from kb0
    const int kb0 = blockIdx.z * A.bsplit;
    const int kcount = min(A.bsplit, nb - kb0);

    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 4 + (XIN ? GemmRoles<PWG>::NCV : 0));
            mbar_init(&empty[s], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&minfull[j], 4 * PWG);
            mbar_init(&minempty[j], 1);
            mbar_init(&tfull[j], 1);
            mbar_init(&tempty[j], 4);
        }
        for (int s = 0; s < GemmCfg<FMT>::BSLOTS; ++s) {
            mbar_init(&bfull[s], 1);
            mbar_init(&bempty[s], 4 * PWG);
        }
        if constexpr (XIN) {
            for (int j = 0; j < 2; ++j) {
                mbar_init(&xfull[j], 1);
                mbar_init(&xempty[j], GemmRoles<PWG>::NCV);
            }
        }
        fence_barrier_init();
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;"
                     :: "r"(smem_u32(tmem_slot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    grid_launch_dependents();
    grid_wait_prior();   // global memory only after the kernels before this one end
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp < EPI_WARP0) {
        // ------------------------------------------------------- producers
        const int t = tid & (GT - 1);          // weight row (and activation row) of the tile
        const int r = r0 + t, i = i0 + t;
        const bool wrow = r < A.n, xrow = i < A.m;
        Q6KRow R, Rn;
        auto load_row = [&](Q6KRow& dst, int b) {
            q6K_row_load(dst, A.w + ((size_t)r * nb + b) * Q6K_BYTES, wrow);
        };
        load_row(R, kb0);
        int b = 0;
        for (; b < kcount && ok; ++b) {
            const int j = b & 1;
            const float dw = half_bits_to_float(R.raw[52]);
            if (b >= 2) {   // slot j's scales are free again
                ok = mbar_wait(&minempty[j], ((b >> 1) - 1) & 1) && mbar_wait(&tempty[j], ((b >> 1) - 1) & 1);
                if (!ok) break;
            }
            {
                float* sj = scl + j * 3 * GT;
                const uint8_t* xb = A.xq + ((size_t)i * nb + kb0 + b) * Q8K_BYTES;
                sj[t] = dw;
                sj[GT + t] = 0.0f;
                sj[2 * GT + t] = xrow ? __ldg(reinterpret_cast<const float*>(xb)) : 0.0f;
            }
            if (b + 1 < kcount) load_row(Rn, kb0 + b + 1);   // next block's bytes, in flight while this one is decoded
            // stage c of the block (c a compile-time constant, so R's fields stay in registers)
            auto stage = [&](auto cc_) -> bool {
                constexpr int c = decltype(cc_)::value;
                const int g = 4 * b + c, s = g % NSTAGE, u = g / NSTAGE;
                if (g >= NSTAGE && !mbar_wait(&empty[s], (u - 1) & 1)) return false;
                uint8_t* st = sm + L::RING + s * L::STAGE;
                if (!XIN && t == 0) {
                    mbar_expect_tx(&full[s], TILE_BYTES);
                    tma_load_2d(st + BOFF, &xmap, (kb0 + b) * QK + c * KS, i0, &full[s]);
                }
                q6K_row_stage(R, c, st, st + TILE_BYTES, t);
                // the ring is shorter than a block: stage c + NSTAGE reuses this
                // slot, so the MMA must have it before the block is finished
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[s]);
                return true;
            };
            using C0 = std::integral_constant<int, 0>;
            using C1 = std::integral_constant<int, 1>;
            using C2 = std::integral_constant<int, 2>;
            using C3 = std::integral_constant<int, 3>;
            ok = stage(C0{}) && stage(C1{}) && stage(C2{}) && stage(C3{});
            if (!ok) break;
            // the block's scales before the epilogue reads them
            __syncwarp();
            if (lane == 0) mbar_arrive(&minfull[j]);
            R = Rn;
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            for (int b = 0; b < kcount && ok; ++b) {
                const int j = b & 1;
                const uint32_t d1 = tmem + j * 256, d2 = d1 + 128;
                if (b >= 2 && !mbar_wait(&tempty[j], ((b >> 1) - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                for (int c = 0; c < 4 && ok; ++c) {
                    const int g = 4 * b + c, s = g % NSTAGE, u = g / NSTAGE;
                    if (!mbar_wait(&full[s], u & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(sm + L::RING + s * L::STAGE);
                    const uint64_t db = umma_desc_sw128(sa + BOFF);
                    const uint64_t dh = umma_desc_sw128(sa), dl = umma_desc_sw128(sa + TILE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {   // K = 16 per MMA: +32 bytes = +2 descriptor units
                        mma_f16(d1, dh + 2 * kk, db + 2 * kk, (c | kk) != 0);
                        mma_f16(d2, dl + 2 * kk, db + 2 * kk, (c | kk) != 0);
                    }
                    mma_commit(&empty[s]);
                }
                if (!ok) break;
                if (!mbar_wait(&minfull[j], (b >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                mma_commit(&minempty[j]);
                mma_commit(&tfull[j]);
            }
        }
        __syncwarp();
    } else if (warp > MMA_WARP) {
        // ------------------------------------------------------- activation converters (XIN)
        if constexpr (XIN) {
            static_assert(!XIN || GemmCfg<FMT>::BSLOTS == 0, "XIN side data: q6_K only in this kernel");
            constexpr int NT = GemmRoles<PWG>::NCV * 32;
            const int u = tid - (MMA_WARP + 1) * 32, cw = u >> 5;
            uint8_t* xst = sm + L::XST;
            if (!A.xtma) {
                xin_zero_tail(xst, min(GT, A.m - i0), u, NT);
                asm volatile("bar.sync 1, %0;" :: "n"(NT) : "memory");
            }
            int nxi = 0;   // warp 0: blocks whose codes were issued
            if (cw == 0)
                for (; nxi < 2 && nxi < kcount; ++nxi)
                    xin_issue(xst + nxi * XSTAGE_BYTES, &xfull[nxi], &xmap, A.xtma != 0, A.xq, nb, A.m, i0, kb0 + nxi, lane);
            int b = 0;
            for (; b < kcount && ok; ++b) {
                const int xs = b & 1;
                if (!mbar_wait(&xfull[xs], (uint32_t)(b >> 1) & 1u)) { ok = false; break; }
                ok = xin_block<NT>(
                    xst + xs * XSTAGE_BYTES, A.xq, nb, i0, kb0 + b, u,
                    [&](int c) {
                        const int g = 4 * b + c;
                        return g < NSTAGE || mbar_wait(&empty[g % NSTAGE], (uint32_t)(g / NSTAGE - 1) & 1u);
                    },
                    [&](int c) { return sm + L::RING + ((4 * b + c) % NSTAGE) * L::STAGE + BOFF; },
                    [&](int c) {
                        fence_async_smem();   // generic writes before the tensor core reads them
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&full[(4 * b + c) % NSTAGE]);
                    });
                if (!ok) break;
                // the staging buffer's reads before its refill
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&xempty[xs]);
                if (cw == 0 && b + 2 < kcount) {
                    if (!mbar_wait(&xempty[xs], (uint32_t)(b >> 1) & 1u)) { ok = false; break; }
                    xin_issue(xst + xs * XSTAGE_BYTES, &xfull[xs], &xmap, A.xtma != 0, A.xq, nb, A.m, i0, kb0 + b + 2, lane);
                    ++nxi;
                }
            }
            // after a wait ran out: let the code copies still in flight land before the CTA exits
            if (!ok && cw == 0 && lane == 0)
                for (int bb = b; bb < nxi; ++bb) (void)mbar_wait(&xfull[bb & 1], (uint32_t)(bb >> 1) & 1u);
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int e = tid - EPI_WARP0 * 32;      // TMEM lane = weight row of the tile
        const int q = warp & 3;                  // this warp's lane quarter
        float acc[GT];
#pragma unroll
        for (int c = 0; c < GT; ++c) acc[c] = 0.0f;
        for (int b = 0; b < kcount && ok; ++b) {
            const int j = b & 1;
            if (!mbar_wait(&tfull[j], (b >> 1) & 1) || !mbar_wait(&minfull[j], (b >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float* sj = scl + j * 3 * GT;
            const float dw = sj[e];
            const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + j * 256;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t v1[16], v2[16];
                tmem_ld16(base + 16 * cc, v1);
                tmem_ld16(base + 128 + 16 * cc, v2);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float dx = sj[2 * GT + 16 * cc + c];
                    // d * (16 D_hi + D_lo)
                    const float tt = __fmul_rn(dw, __fmaf_rn(16.0f, __uint_as_float(v1[c]), __uint_as_float(v2[c])));
                    acc[16 * cc + c] = __fmaf_rn(dx, tt, acc[16 * cc + c]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[j]);
        }
        const int r = r0 + e;
        float* out = A.part ? A.part + (size_t)blockIdx.z * A.m * A.n : A.y;
        if (r < A.n) {
#pragma unroll
            for (int c = 0; c < GT; ++c)
                if (i0 + c < A.m) out[(size_t)(i0 + c) * A.n + r] = acc[c];
        }
    }
    if (!ok && lane == 0) atomicOr(A.fault, 2u);
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem) : "memory");
    }
}

// ---------------------------------------------------------------------------
// q4_K / q5_K with the A operand in tensor memory.  The producers decode each
// 64-wide K stage of their weight row straight into a ring of four 32-column
// tensor-memory stages (tcgen05.st), and the MMA reads A from there
// (tcgen05.mma [d], [a], b-desc): shared memory carries only the activation
// tiles (TMA) and the per-block min operands, half the traffic of an A tile
// in shared memory.  Tensor memory (512 columns): D1 (isum) double-buffered
// at columns 0 and 128, D2 (msum) single-buffered at 256, the A ring at
// 384 + 32 s.  The epilogue drains D1 and D2 of a block together and then
// releases both.  Roles: warps 0-7 producers (two warpgroups, stages 2h,
// 2h + 1 of every block), warps 8-15 epilogue (warp e: TMEM lanes 32 (e % 4)
// .., activation columns 64 (e / 4) .. + 63), warp 16 issues the MMAs.  No
// register hand-over: 17 warps at 96.
// The MMA thread waits as seldom as it can: an mbarrier wait takes a few
// hundred cycles even when the phase is complete, and the tensor pipe's
// instruction queue is short, so each wait leaves the pipe idle for a while.
// Each producer warpgroup publishes its two stages (and their activation
// tiles) on one barrier; the second warpgroup's barrier also covers the min
// operands, written and fenced before it.  Four waits a block: D1's slot, the
// two halves, D2.  (XIN keeps a barrier per stage: its converters finish the
// B tiles one stage at a time.)  The weight blocks come through a four-slot
// TMA ring.
// XIN (no workspace): warps 17-19 widen the activation codes from xq into
// the B tiles and write the side data into the block slots (xin_issue,
// xin_convert, xin_side_store) in place of the TMA; 20 warps keep five per
// sub-partition, so the register budget stays at 96.
// ---------------------------------------------------------------------------
constexpr int TM_EPI_WARP0 = 8, TM_MMA_WARP = 16, TM_NSTAGE = 4;
constexpr int TM_NCV = 3;   // converter warps (XIN)
constexpr int tm_threads(bool xin) { return (TM_MMA_WARP + 1 + (xin ? TM_NCV : 0)) * 32; }
constexpr uint32_t TM_D1 = 0, TM_D2 = 256, TM_A = 384;
// slots of the ring of weight blocks: block b + slots is requested once block b
// is decoded (the form with the widening converters has room for two)
__host__ __device__ constexpr int tm_bslots(bool xin) { return xin ? 2 : 4; }

template <int FMT, bool XIN>
struct TmSmem {
    static constexpr int RING = 0;                                            // B tiles, 4 x 16 KB
    static constexpr int MIN = RING + TM_NSTAGE * TILE_BYTES;                 // 2 x 16 KB (none for q6_K)
    static constexpr int SCL = MIN + (FMT == Q6TM ? 0 : 2 * TILE_BYTES);      // 2 x (d, dmin, dx) x 128 f32
    static constexpr int WT = GT * GemmCfg<FMT>::WPITCH;
    static constexpr int BTX = WT + GT * AUXB;
    static constexpr int BSLOT = (BTX + 1023) & ~1023;
    static constexpr int BRING = (SCL + 2 * 3 * GT * 4 + 1023) & ~1023;
    static constexpr int XST = BRING + tm_bslots(XIN) * BSLOT;                // XIN: 2 staging buffers
    static constexpr int BAR = XST + (XIN ? 2 * XSTAGE_BYTES : 0);
    static constexpr int NBAR = 2 * TM_NSTAGE + 8 + 2 * tm_bslots(XIN) + 1 + (XIN ? 4 : 0);
    static constexpr int TMEMP = BAR + NBAR * 8;
    static constexpr int BYTES = TMEMP + 16;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void mma_f16_ta(uint32_t dtmem, uint32_t atmem, uint64_t db, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(dtmem), "r"(atmem), "l"(db), "r"(IDESC_F16_128x128), "r"(accumulate));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
                 "%15,%16};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                    "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                    "r"(r[15]) : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
                 "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                    "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                    "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
                    "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
                    "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}

template <int FMT, bool XIN, bool GATE>
__global__ void __launch_bounds__(tm_threads(XIN), 1) gemm_tm_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                const __grid_constant__ CUtensorMap wmap,
                                                                const __grid_constant__ CUtensorMap amap,
                                                                const GemmArgs A) {
    using L = TmSmem<FMT, XIN>;
    constexpr int NSTAGE = TM_NSTAGE, NBS = tm_bslots(XIN);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    // full[c]: stage c's A rows (4 producer-warp arrivals) and B tile (TMA bytes; XIN: converter warps).
    // Without XIN the two stages of a producer half share one barrier, full[c & 2] (the half publishes
    // them together); with XIN the converters finish the B tiles one stage at a time, so each has its own.
    constexpr bool MERGE = !XIN;
    uint64_t* full = bars;                  // [4]
    uint64_t* empty = bars + NSTAGE;        // [4]: MMA commit (frees the TMEM A stage and the B tile)
    uint64_t* minfull = bars + 2 * NSTAGE;  // [2]: 8 producer-warp arrivals (min operands, scales)
    uint64_t* minempty = minfull + 2;       // [2]: MMA commit
    uint64_t* tfull = minfull + 4;          // [2]: MMA commit
    uint64_t* tempty = minfull + 6;         // [2]: 8 epilogue-warp arrivals
    uint64_t* bfull = minfull + 8;          // [NBS]: TMA bytes of a weight block and its side data (XIN: + converter warps)
    uint64_t* bempty = bfull + NBS;         // [NBS]: 8 producer-warp arrivals
    uint64_t* d2free = bempty + NBS;        // [1]: 8 epilogue-warp arrivals once D2 is read
    uint64_t* xfull = d2free + 1;           // XIN [2]: bulk-copy bytes of a staged block of codes
    uint64_t* xempty = xfull + 2;           // XIN [2]: converter-warp arrivals once it is widened
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::TMEMP);
    float* scl = reinterpret_cast<float*>(sm + L::SCL);   // [2][3][128]: d, dmin, dx

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's tile: weight rows from r0, activation rows from i0, K blocks [kb0, kb0 + kcount)
    // x: activation tile, y: weight tile, so the CTAs that share a weight tile
    // run next to each other and its re-reads come from L2
    const int r0 = (blockIdx.y + A.ty0) * GT, i0 = blockIdx.x * GT;
    const int nb = A.nb;
    const int kb0 = blockIdx.z * A.bsplit;
    const int kcount = min(A.bsplit, nb - kb0);

    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 4 + (XIN ? TM_NCV : 0));
            mbar_init(&empty[s], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&minfull[j], 8);
            mbar_init(&minempty[j], 1);
            mbar_init(&tfull[j], 1);
            mbar_init(&tempty[j], 8);
        }
        for (int s = 0; s < NBS; ++s) {
            mbar_init(&bfull[s], 1 + (XIN ? TM_NCV : 0));
            mbar_init(&bempty[s], 8);
        }
        mbar_init(d2free, 8);
        if constexpr (XIN) {
            for (int j = 0; j < 2; ++j) {
                mbar_init(&xfull[j], 1);
                mbar_init(&xempty[j], TM_NCV);
            }
        }
        fence_barrier_init();
    }
    if (warp == TM_MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;"
                     :: "r"(smem_u32(tmem_slot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    grid_launch_dependents();
    grid_wait_prior();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp < TM_EPI_WARP0) {
        // ------------------------------------------------------- producers
        const int t = tid & (GT - 1);          // weight row (and activation row) of the tile
        const int half = warp >> 2;            // stages 2 half, 2 half + 1 of every block
        const uint32_t alane = (uint32_t)((warp & 3) * 32) << 16;
        using Row = typename std::conditional<
            FMT == Q6TM, Q6Half, typename std::conditional<FMT <= 3, QlowHalf<FMT>, QxKHalf<FMT>>::type>::type;
        constexpr int WROW = GemmCfg<FMT>::WROW, WPITCH = GemmCfg<FMT>::WPITCH;
        Row R;
        int nissued = 0;
        auto issue_block = [&](int bb) {   // thread 0: block bb of the tile into slot bb % NBS
            ++nissued;
            const int s = bb % NBS;
            uint8_t* dst = sm + L::BRING + s * L::BSLOT;
            mbar_arrive_expect_tx(&bfull[s], (uint32_t)(XIN ? L::WT : L::BTX));
            tma_load_2d(dst, &wmap, ((kb0 + bb) * WROW) & ~15, r0, &bfull[s]);   // the block's 16-byte window
            if constexpr (!XIN) tma_load_2d(dst + L::WT, &amap, (kb0 + bb) * AUXB, i0, &bfull[s]);
        };
        if (tid == 0)
            for (int bb = 0; bb < NBS && bb < kcount; ++bb) issue_block(bb);
        int gb = 0;   // block of the tile: slots and phases
        {
            for (int b = 0; b < kcount && ok; ++b, ++gb) {
                const int j = gb & 1;
                uint32_t bsw[8];
                float dx;
                {
                    const int s = gb % NBS;
                    if (!mbar_wait(&bfull[s], (uint32_t)(gb / NBS) & 1u)) { ok = false; break; }
                    const uint8_t* slot = sm + L::BRING + s * L::BSLOT;
                    if constexpr (FMT == Q6TM) {
                        q6_half_load(R, slot + t * WPITCH, ((kb0 + b) * WROW) & 15, half);
                    } else if constexpr (FMT <= 3) {
                        qlow_half_load<FMT>(R, slot + t * WPITCH, ((kb0 + b) * WROW) & 15, half);
                    } else {
                        qxK_half_load<FMT>(R, slot + t * WPITCH, half);
                    }
                    const uint4* ax = reinterpret_cast<const uint4*>(slot + L::WT + t * AUXB);
                    const uint4 a0 = ax[0], a1 = ax[1], a2 = ax[2];
                    bsw[0] = a0.x; bsw[1] = a0.y; bsw[2] = a0.z; bsw[3] = a0.w;
                    bsw[4] = a1.x; bsw[5] = a1.y; bsw[6] = a1.z; bsw[7] = a1.w;
                    dx = __uint_as_float(a2.x);
                    fence_async_smem();   // these reads before the slot's refill by TMA
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bempty[s]);
                }
                if constexpr (FMT == 4 || FMT == 5) qxK_half_prepare<FMT>(R, half);
                if (gb >= 2) {   // slot j's min operands and scales are free again
                    ok = mbar_wait(&minempty[j], ((gb >> 1) - 1) & 1) && mbar_wait(&tempty[j], ((gb >> 1) - 1) & 1);
                    if (!ok) break;
                }
                if (half == 1) {
                    if constexpr (FMT != Q6TM) {
                    // min operands: K 0..15 the weight row's mins m_(g/2); K 16..31 the activation row's bsums
                    uint8_t* mt = sm + L::MIN + j * TILE_BYTES;
                    uint32_t mv[8];
                    if constexpr (FMT <= 3)
                        qlow_half_min_pairs<FMT>(R, mv);
                    else
                        qxK_min_pairs(R.hdr, mv);
                    *reinterpret_cast<uint4*>(mt + sw128_chunk(t, 0)) = make_uint4(mv[0], mv[1], mv[2], mv[3]);
                    *reinterpret_cast<uint4*>(mt + sw128_chunk(t, 1)) = make_uint4(mv[4], mv[5], mv[6], mv[7]);
                    *reinterpret_cast<uint4*>(mt + sw128_chunk(t, 2)) = make_uint4(bsw[0], bsw[1], bsw[2], bsw[3]);
                    *reinterpret_cast<uint4*>(mt + sw128_chunk(t, 3)) = make_uint4(bsw[4], bsw[5], bsw[6], bsw[7]);
                    }
                } else {
                    float* sj = scl + j * 3 * GT;
                    sj[t] = R.d;
                    if constexpr (FMT != Q6TM) sj[GT + t] = R.dmin;
                    sj[2 * GT + t] = dx;
                }
                // the block's two stages of this warpgroup, c = 2 half + CL: A into tensor
                // memory, B by TMA (CL a compile-time constant, so R's fields stay in registers)
                auto stage = [&](auto cl_) -> bool {
                    constexpr int CL = decltype(cl_)::value;
                    const int c = 2 * half + CL;   // stage, and its ring slot (one block long)
                    if (gb >= 1) {
                        if (!mbar_wait(&empty[c], (uint32_t)(gb - 1) & 1u)) return false;
                        tc_fence_after();
                    }
                    if (!XIN && t == 0) {   // the half's barrier counts both of its stages' tiles
                        mbar_expect_tx(&full[c & 2], TILE_BYTES);
                        tma_load_2d(sm + L::RING + c * TILE_BYTES, &xmap, (kb0 + b) * QK + c * KS, i0, &full[c & 2]);
                    }
                    if constexpr (FMT == Q6TM) {
                        // two operands (16 hi (q - 32) at columns 256 .., lo (q - 32) at 384 ..), 16 columns at a time
                        uint32_t vh[16], vl[16];
                        q6_half_stage_regs<CL, 0>(R, half, vh, vl);
                        tmem_st16(tmem + alane + TM_D2 + 32 * c, vh);
                        tmem_st16(tmem + alane + TM_A + 32 * c, vl);
                        q6_half_stage_regs<CL, 1>(R, half, vh, vl);
                        tmem_st16(tmem + alane + TM_D2 + 32 * c + 16, vh);
                        tmem_st16(tmem + alane + TM_A + 32 * c + 16, vl);
                    } else {
                        uint32_t v[32];
                        if constexpr (FMT <= 3)
                            qlow_half_stage_regs<FMT, CL>(R, half, v);
                        else
                            qxK_half_stage_regs<FMT, CL>(R, c, v);
                        tmem_st32(tmem + alane + TM_A + 32 * c, v);
                    }
                    return true;
                };
                using C0 = std::integral_constant<int, 0>;
                using C1 = std::integral_constant<int, 1>;
                ok = stage(C0{}) && stage(C1{});
                if (!ok) break;
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                fence_async_smem();   // min operands and scales before the MMA / epilogue read them
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&minfull[j]);
                    mbar_arrive(&full[2 * half]);
                    if constexpr (!MERGE) mbar_arrive(&full[2 * half + 1]);
                }
                // refill this block's weight slot once every producer warp has read it
                if (tid == 0 && b + NBS < kcount) {
                    if (!mbar_wait(&bempty[gb % NBS], (uint32_t)(gb / NBS) & 1u)) { ok = false; break; }
                    issue_block(b + NBS);
                }
            }
        }
        // after a wait ran out: let this CTA's weight copies still in flight land before it exits
        if (!ok && tid == 0)
            for (int bb = gb; bb < nissued; ++bb) (void)mbar_wait(&bfull[bb % NBS], (uint32_t)(bb / NBS) & 1u);
    } else if (warp == TM_MMA_WARP) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int gb = 0;
            {
                for (int b = 0; b < kcount && ok; ++b, ++gb) {
                    const int j = gb & 1;
                    const uint32_t d1 = tmem + TM_D1 + 128 * j;
                    if (gb >= 2 && !mbar_wait(&tempty[j], ((gb >> 1) - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    for (int c = 0; c < 4 && ok; ++c) {
                        // without XIN, one wait per producer half: its two stages are published together
                        if (!MERGE || (c & 1) == 0) {
                            if (!mbar_wait(&full[c], (uint32_t)gb & 1u)) { ok = false; break; }
                            tc_fence_after();
                        }
                        const uint64_t db = umma_desc_sw128(smem_u32(sm + L::RING + c * TILE_BYTES));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {  // K = 16 per MMA: 8 TMEM columns, +2 descriptor units
                            if constexpr (FMT == Q6TM) {   // both parts of the scale into the one accumulator
                                mma_f16_ta(d1, tmem + TM_D2 + 32 * c + 8 * kk, db + 2 * kk, (c | kk) != 0);
                                mma_f16_ta(d1, tmem + TM_A + 32 * c + 8 * kk, db + 2 * kk, 1u);
                            } else {
                                mma_f16_ta(d1, tmem + TM_A + 32 * c + 8 * kk, db + 2 * kk, (c | kk) != 0);
                            }
                        }
                        mma_commit(&empty[c]);
                    }
                    if (!ok) break;
                    // the min operands were written (and fenced) before the second half's
                    // stages were published, so the wait on full[2] (or full[3]) covers them
                    if constexpr (FMT != Q6TM) {   // q6_K: no min term
                        if (gb >= 1 && !mbar_wait(d2free, (uint32_t)(gb - 1) & 1u)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t ma = smem_u32(sm + L::MIN + j * TILE_BYTES);
                        mma_f16(tmem + TM_D2, umma_desc_sw128(ma), umma_desc_sw128(ma) + 2, 0u);
                    }
                    mma_commit(&minempty[j]);
                    mma_commit(&tfull[j]);
                }
            }
        }
        __syncwarp();
    } else if (warp > TM_MMA_WARP) {
        // ------------------------------------------------------- activation converters (XIN)
        if constexpr (XIN) {
            static_assert(NBS == 2, "the converters index the weight-block ring in pairs");
            constexpr int NT = TM_NCV * 32;
            const int u = tid - (TM_MMA_WARP + 1) * 32, cw = u >> 5;
            uint8_t* xst = sm + L::XST;
            if (!A.xtma) {
                xin_zero_tail(xst, min(GT, A.m - i0), u, NT);
                asm volatile("bar.sync 1, %0;" :: "n"(NT) : "memory");
            }
            int nxi = 0;   // warp 0: blocks whose codes were issued
            if (cw == 0)
                for (; nxi < 2 && nxi < kcount; ++nxi)
                    xin_issue(xst + nxi * XSTAGE_BYTES, &xfull[nxi], &xmap, A.xtma != 0, A.xq, nb, A.m, i0, kb0 + nxi, lane);
            XinSide<NT> sd;
            xin_side_load(sd, A.xq, nb, A.m, i0, kb0, u);
            int gb = 0;
            for (int b = 0; b < kcount && ok; ++b, ++gb) {
                const int s = gb & 1, blk = kb0 + b;
                // the block's side data into its weight slot, the next block's into registers
                if (gb >= 2 && !mbar_wait(&bempty[s], (uint32_t)((gb >> 1) - 1) & 1u)) { ok = false; break; }
                xin_side_store(sd, sm + L::BRING + s * L::BSLOT + L::WT, u);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bfull[s]);
                if (b + 1 < kcount) xin_side_load(sd, A.xq, nb, A.m, i0, blk + 1, u);
                // the four B stages, each once the MMA has finished the previous block's
                if (!mbar_wait(&xfull[s], (uint32_t)(gb >> 1) & 1u)) { ok = false; break; }
                ok = xin_block<NT>(
                    xst + s * XSTAGE_BYTES, A.xq, nb, i0, blk, u,
                    [&](int c) { return gb == 0 || mbar_wait(&empty[c], (uint32_t)(gb - 1) & 1u); },
                    [&](int c) { return sm + L::RING + c * TILE_BYTES; },
                    [&](int c) {
                        fence_async_smem();   // generic writes before the tensor core reads them
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&full[c]);
                    });
                if (!ok) break;
                // the staging buffer's reads before its refill
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&xempty[s]);
                if (cw == 0 && b + 2 < kcount) {
                    if (!mbar_wait(&xempty[s], (uint32_t)(gb >> 1) & 1u)) { ok = false; break; }
                    xin_issue(xst + s * XSTAGE_BYTES, &xfull[s], &xmap, A.xtma != 0, A.xq, nb, A.m, i0, blk + 2, lane);
                    ++nxi;
                }
            }
            // after a wait ran out: let the code copies still in flight land before the CTA exits
            if (!ok && cw == 0 && lane == 0)
                for (int bb = gb; bb < nxi; ++bb) (void)mbar_wait(&xfull[bb & 1], (uint32_t)(bb >> 1) & 1u);
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int e = warp - TM_EPI_WARP0;
        const int q = e & 3, chalf = e >> 2;     // TMEM lane quarter, activation-column half
        const int row = 32 * q + lane;           // weight row of the tile
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        int gb = 0;
        {
            uint64_t acc2[32];   // columns 2c, 2c + 1 as f32 pairs (packed f32x2 arithmetic)
#pragma unroll
            for (int c = 0; c < 32; ++c) acc2[c] = 0ull;
            for (int b = 0; b < kcount && ok; ++b, ++gb) {
                const int j = gb & 1;
                if (!mbar_wait(&tfull[j], (gb >> 1) & 1) || !mbar_wait(&minfull[j], (gb >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float* sj = scl + j * 3 * GT;
                const float dw = sj[row], dmw = FMT == Q6TM ? 0.0f : sj[GT + row];
                const uint64_t dw2 = f2_pack(dw, dw), ndmw2 = f2_pack(-dmw, -dmw);
                const uint64_t* dxv = reinterpret_cast<const uint64_t*>(sj + 2 * GT + 64 * chalf);
                // D1 and D2 together: + dx * (d * isum - dmin * msum), two columns per
                // instruction, each rounded as fma(dx, fma(d, isum, (-dmin) * msum), acc)
                // CH columns per tensor-memory load (the form without the widening
                // converters has the registers for fewer, longer-lived loads: 4)
                constexpr int CH = XIN ? 8 : 4;
#pragma unroll
                for (int cc = 0; cc < 64 / CH; ++cc) {
                    uint32_t v1[CH], v2[CH];
                    if constexpr (FMT != Q6TM) tmem_ld_n(tl + TM_D2 + 64 * chalf + CH * cc, v2);
                    tmem_ld_n(tl + TM_D1 + 128 * j + 64 * chalf + CH * cc, v1);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int c = 0; c < CH / 2; ++c) {
                        const uint64_t i2 = f2_pack(__uint_as_float(v1[2 * c]), __uint_as_float(v1[2 * c + 1]));
                        uint64_t t;
                        if constexpr (FMT == Q6TM) {
                            t = mul_f32x2(dw2, i2);
                        } else {
                            const uint64_t m2 = f2_pack(__uint_as_float(v2[2 * c]), __uint_as_float(v2[2 * c + 1]));
                            t = fma_f32x2(dw2, i2, mul_f32x2(ndmw2, m2));
                        }
                        acc2[CH / 2 * cc + c] = fma_f32x2(dxv[CH / 2 * cc + c], t, acc2[CH / 2 * cc + c]);
                    }
                }
                // both accumulators read: D2 for the next block's min MMA, D1 for the block after
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(d2free);
                    mbar_arrive(&tempty[j]);
                }
            }
            float acc[64];
#pragma unroll
            for (int c = 0; c < 32; ++c) f2_unpack(acc2[c], acc[2 * c], acc[2 * c + 1]);
            const int r = r0 + row;
            float* out = A.part ? A.part + (size_t)blockIdx.z * A.m * A.n : A.y;
            if (A.csplit > 1) {
                // cluster K split: this CTA's partial tile into its B ring (idle once the last
                // block's MMAs are done), four columns per 16 bytes, thread-major
                float4* red = reinterpret_cast<float4*>(sm + L::RING) + e * 32 + lane;
#pragma unroll
                for (int c4 = 0; c4 < 16; ++c4)
                    red[c4 * 256] = make_float4(acc[4 * c4], acc[4 * c4 + 1], acc[4 * c4 + 2], acc[4 * c4 + 3]);
            } else if (ok && r < A.n) {
                if constexpr (GATE) {
                    // SwiGLU pair: the gate GEMM's result for the same element, 16 loads at a time
#pragma unroll
                    for (int cb = 0; cb < 64; cb += 16) {
                        float g[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int i = i0 + 64 * chalf + cb + c;
                            g[c] = i < A.m ? A.gate[(size_t)i * A.n + r] : 0.0f;
                        }
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int i = i0 + 64 * chalf + cb + c;
                            if (i < A.m) out[(size_t)i * A.n + r] = swiglu1(g[c], acc[cb + c]);
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int i = i0 + 64 * chalf + c;
                        if (i < A.m) out[(size_t)i * A.n + r] = acc[c];
                    }
                }
            }
        }
    }
    if (!ok && lane == 0) atomicOr(A.fault, 2u);
    tc_fence_before();
    __syncthreads();
    if (A.csplit > 1) {
        // every thread of every CTA of the cluster passes both barriers: the partials
        // are visible, rank 0 adds them in rank order (the same bits every run) and
        // stores the tile, and no CTA leaves while its shared memory is still read
        cluster_sync_all();
        if (cluster_rank() == 0 && warp >= TM_EPI_WARP0 && warp < TM_MMA_WARP) {
            const int e = warp - TM_EPI_WARP0, q = e & 3, chalf = e >> 2;
            const int r = r0 + 32 * q + lane;
            const float4* red = reinterpret_cast<const float4*>(sm + L::RING) + e * 32 + lane;
            if (r < A.n) {
#pragma unroll 4
                for (int c4 = 0; c4 < 16; ++c4) {
                    float4 v = red[c4 * 256];
                    for (int z = 1; z < A.csplit; ++z) {
                        const float4 u = ld_peer_f4(red + c4 * 256, (uint32_t)z);
                        v.x = __fadd_rn(v.x, u.x);
                        v.y = __fadd_rn(v.y, u.y);
                        v.z = __fadd_rn(v.z, u.z);
                        v.w = __fadd_rn(v.w, u.w);
                    }
                    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int i = i0 + 64 * chalf + 4 * c4 + t;
                        if (i < A.m) {
                            if constexpr (GATE)
                                A.y[(size_t)i * A.n + r] = swiglu1(A.gate[(size_t)i * A.n + r], vv[t]);
                            else
                                A.y[(size_t)i * A.n + r] = vv[t];
                        }
                    }
                }
            }
        }
        __syncwarp();
        cluster_sync_all();
    }
    if (warp == TM_MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem) : "memory");
    }
}

// q8_K codes -> f16 activation matrix [m][k] (the GEMM's B operand source),
// and per block the side data the producers take by TMA: the bsums as f16
// pairs, d and three zero words (AUXB bytes)
__global__ void gemm_x16_kernel(const uint8_t* __restrict__ xq, __half* __restrict__ x16, uint32_t* __restrict__ aux,
                                long long nblocks) {
    grid_launch_dependents();
    grid_wait_prior();
    const long long total = nblocks * 32;                 // 8 codes per item
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
         it += (long long)gridDim.x * blockDim.x) {
        const long long blk = it >> 5;
        const int part = (int)(it & 31);
        const uint32_t* src = reinterpret_cast<const uint32_t*>(xq + blk * Q8K_BYTES + 4) + 2 * part;
        const uint32_t a = __ldg(src), c = __ldg(src + 1);
        uint32_t o[4];
        const uint32_t wv[2] = {a, c};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t v = wv[h];
            o[2 * h] = h2_bits(__halves2half2(__int2half_rn((int)(int8_t)(v & 0xFF)),
                                              __int2half_rn((int)(int8_t)((v >> 8) & 0xFF))));
            o[2 * h + 1] = h2_bits(__halves2half2(__int2half_rn((int)(int8_t)((v >> 16) & 0xFF)),
                                                  __int2half_rn((int)(int8_t)(v >> 24))));
        }
        *reinterpret_cast<uint4*>(x16 + blk * QK + 8 * part) = make_uint4(o[0], o[1], o[2], o[3]);
        if (part < AUXB / 4) {
            const uint8_t* blkp = xq + blk * Q8K_BYTES;
            uint32_t v = 0;
            if (part < 8) {   // bsums 2 part, 2 part + 1 as an f16 pair (|bsum| <= 2048: exact)
                const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(blkp + 260) + part);
                v = h2_bits(__halves2half2(__int2half_rn((int)(int16_t)(u & 0xFFFF)),
                                           __int2half_rn((int)(int16_t)(u >> 16))));
            }
            else if (part == 8)
                v = __ldg(reinterpret_cast<const uint32_t*>(blkp));
            aux[blk * (AUXB / 4) + part] = v;
        }
    }
}

// SwiGLU of a gate/up pair: h = silu(h) * u = h / (1 + e^-h) * u, elementwise
// (h holds the gate GEMM's output on entry).
__global__ void gemm_swiglu_kernel(float* __restrict__ h, const float* __restrict__ u, long long count) {
    grid_launch_dependents();
    grid_wait_prior();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x) {
        h[i] = swiglu1(h[i], u[i]);
    }
}

// Split K: y = the splits' partial sums, added in split order (deterministic).
__global__ void gemm_split_reduce_kernel(const float* __restrict__ part, float* __restrict__ y, long long count,
                                         int splits) {
    grid_launch_dependents();
    grid_wait_prior();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x) {
        float s = part[i];
        for (int z = 1; z < splits; ++z) s = __fadd_rn(s, part[(size_t)z * count + i]);
        y[i] = s;
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// f16 activation codes [m][k], then the side data [m][k/256][AUXB bytes]
static size_t gemm_x16_bytes(long long m, int k) { return (((size_t)m * k * 2) + 255) & ~(size_t)255; }
size_t gemm_workspace_bytes(long long m, int k) {
    return gemm_x16_bytes(m, k) + ((((size_t)m * (k / QK) * AUXB) + 255) & ~(size_t)255);
}

// K splits when the output tiles alone leave most SMs idle: as many as fill
// the SMs once, each split at least four 256-weight blocks long.
static int gemm_splits(long long m, int n, int nb) {
    const long long tiles = (long long)((n + GT - 1) / GT) * ((m + GT - 1) / GT);
    long long s = num_sms() / (tiles > 0 ? tiles : 1);
    if (s > nb / 4) s = nb / 4;
    return s > 1 ? (int)s : 1;
}

static size_t gemm_split_bytes(long long m, int n, int splits) {
    return splits > 1 ? (size_t)splits * m * n * sizeof(float) : 0;
}

// ws == nullptr: the XIN kernels (activation codes widened in the kernel, no
// pre-pass, no K split, nothing allocated).  Otherwise the pre-pass writes
// the f16 activations and side data into ws for the TMA, and K is split when
// ws also holds the partial sums.  gate: see GemmArgs (unsplit q4_K only).
template <int FMT>
static cudaError_t gemm_tc(const uint8_t* w, const uint8_t* xq, float* y, long long m, int n, int k, void* ws,
                           size_t ws_bytes, const float* gate, cudaStream_t stream) {
    const int nb = k / QK;
    const bool xin = ws == nullptr;
    int splits = 1;
    float* part = nullptr;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap map, wmap, amap;   // unused ones stay zero and are never read
    memset(&map, 0, sizeof(map));
    memset(&wmap, 0, sizeof(wmap));
    memset(&amap, 0, sizeof(amap));
    bool xtma = false;
    if (xin && nb % 4 == 0 && ((uintptr_t)xq & 15u) == 0) {
        // the q8_K rows as four-byte words: a box of 128 rows x XROW bytes
        const cuuint64_t dims[2] = {(cuuint64_t)nb * (Q8K_BYTES / 4), (cuuint64_t)m};
        const cuuint64_t strides[1] = {(cuuint64_t)nb * Q8K_BYTES};
        const cuuint32_t box[2] = {(cuuint32_t)(XROW / 4), (cuuint32_t)GT};
        xtma = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(xq), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        if (!xtma) memset(&map, 0, sizeof(map));
    }
    if (!xin) {
        __half* x16 = static_cast<__half*>(ws);
        uint32_t* aux = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + gemm_x16_bytes(m, k));
        // split K only when the caller's workspace holds the partial sums too
        if (!gate) splits = gemm_splits(m, n, nb);
        if (ws_bytes < gemm_workspace_bytes(m, k) + gemm_split_bytes(m, n, splits)) splits = 1;
        if (splits > 1) part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + gemm_workspace_bytes(m, k));
        const long long nblocks = m * nb;
        long long grid = (nblocks * 32 + 255) / 256;
        const long long cap = (long long)num_sms() * 8;
        if (grid > cap) grid = cap;
        cudaError_t e = launch_kernel(gemm_x16_kernel, dim3((unsigned)grid), dim3(256), 0, stream, xq, x16, aux,
                                      nblocks);
        if (e != cudaSuccess) return e;
        const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)m};
        const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
        const cuuint32_t box[2] = {(cuuint32_t)KS, (cuuint32_t)GT};
        if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x16, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if constexpr (GemmCfg<FMT>::BSLOTS > 0) {
            // the side data: rows of nb * AUXB bytes, a box is one block of 128 activation rows
            const cuuint64_t ad[2] = {(cuuint64_t)nb * AUXB, (cuuint64_t)m};
            const cuuint64_t as_[1] = {(cuuint64_t)nb * AUXB};
            const cuuint32_t ab[2] = {(cuuint32_t)AUXB, (cuuint32_t)GT};
            if (enc(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, aux, ad, as_, ab, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
    }
    // the tensor-memory kernels (q2_K .. q6_K): the raw weight blocks (rows of nb * WROW bytes; a box is
    // one block's 16-byte-aligned window, WPITCH bytes, of 128 rows; rows past
    // n and bytes past a row's end read as zeros)
    if constexpr (GemmCfg<FMT>::BSLOTS > 0) {
        constexpr int WROW = GemmCfg<FMT>::WROW;
        const cuuint64_t wd[2] = {(cuuint64_t)nb * WROW, (cuuint64_t)n};
        const cuuint64_t ws_[1] = {(cuuint64_t)nb * WROW};
        const cuuint32_t wb[2] = {(cuuint32_t)GemmCfg<FMT>::WPITCH, (cuuint32_t)GT};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), wd, ws_, wb, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    GemmArgs A;
    A.w = w;
    A.xq = xq;
    A.y = y;
    A.gate = gate;
    A.xtma = xtma ? 1 : 0;
    A.csplit = 1;
    A.ty0 = 0;
    A.fault = fault_word();
    if (!A.fault) return cudaErrorInvalidDevicePointer;
    A.m = (int)m;
    A.n = n;
    A.nb = nb;
    A.part = part;
    A.bsplit = (nb + splits - 1) / splits;
    splits = (nb + A.bsplit - 1) / A.bsplit;   // no empty split
    const dim3 grid((unsigned)((m + GT - 1) / GT), (unsigned)((n + GT - 1) / GT), (unsigned)splits);
    auto run = [&](auto kernel, int threads, int smem) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        return launch_kernel(kernel, grid, dim3(threads), smem, stream, map, wmap, amap, A);
    };
    // Many output tiles, unsplit: when the grid's last wave would hold at most
    // half the SMs' worth of tiles, the weight-tile rows that make it up run as
    // a second launch after the others, K split over a cluster of up to four
    // CTAs per tile (partial tiles added through distributed shared memory), so
    // that wave takes a fraction of a tile's time.  The split changes the f32
    // order of those rows only; the same shape always splits the same way.
    auto run_tail = [&](auto kernel, int threads, int smem) -> cudaError_t {
        const long long S = num_sms(), X = grid.x, Y = grid.y, tiles = X * Y;
        if (grid.z == 1 && tiles > S) {
            const long long waves = tiles / S, rem = tiles - waves * S, ymain = waves * S / X;
            if (rem > 0 && rem <= S / 2 && ymain > 0 && ymain < Y) {
                const long long ytail = Y - ymain;
                long long want = S / (X * ytail);
                if (want > 4) want = 4;
                if (want > nb / 4) want = nb / 4;
                for (int cz = (int)want; cz >= 2; --cz) {
                    const int bs = (nb + cz - 1) / cz;
                    const int z = (nb + bs - 1) / bs;   // no empty split
                    const dim3 gt(grid.x, (unsigned)ytail, (unsigned)z);
                    if (z < 2 || max_active_clusters(kernel, gt, dim3(threads), (size_t)smem, (unsigned)z) < 1)
                        continue;
                    cudaError_t e = launch_kernel(kernel, dim3(grid.x, (unsigned)ymain, 1), dim3(threads), smem,
                                                  stream, map, wmap, amap, A);
                    if (e != cudaSuccess) return e;
                    GemmArgs T = A;
                    T.ty0 = (int)ymain;
                    T.bsplit = bs;
                    T.csplit = z;
                    return launch_kernel_cluster(kernel, gt, dim3(threads), smem, stream, (unsigned)z, map, wmap,
                                                 amap, T);
                }
            }
        }
        return launch_kernel(kernel, grid, dim3(threads), smem, stream, map, wmap, amap, A);
    };
    // the tensor-memory kernels without a workspace split: the tail above
    auto run_tm = [&](auto kernel, int threads, int smem) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        return run_tail(kernel, threads, smem);
    };
    // the tensor-memory kernels without a workspace: few output tiles, split K over a
    // cluster of up to eight CTAs per tile (partial tiles added through distributed
    // shared memory); many tiles, the short last wave as above
    auto run_cluster = [&](auto kernel, int threads, int smem) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int want = gemm_splits(m, n, nb);
        if (want > 8) want = 8;
        for (int cz = want; cz >= 2; --cz) {
            const int bs = (nb + cz - 1) / cz;
            const int z = (nb + bs - 1) / bs;   // no empty split
            const dim3 g(grid.x, grid.y, (unsigned)z);
            if (z < 2 || max_active_clusters(kernel, g, dim3(threads), (size_t)smem, (unsigned)z) < 1) continue;
            GemmArgs B = A;
            B.bsplit = bs;
            B.csplit = z;
            return launch_kernel_cluster(kernel, g, dim3(threads), smem, stream, (unsigned)z, map, wmap, amap, B);
        }
        return run_tail(kernel, threads, smem);
    };
    cudaError_t e;
    if constexpr (FMT != 6) {
        if (gate) {
            if (FMT != 4 || !xin) return cudaErrorInvalidValue;
            e = run_cluster(gemm_tm_kernel<4, true, true>, tm_threads(true), TmSmem<4, true>::ALLOC);
        } else {
            e = xin ? run_cluster(gemm_tm_kernel<FMT, true, false>, tm_threads(true), TmSmem<FMT, true>::ALLOC)
                    : run_tm(gemm_tm_kernel<FMT, false, false>, tm_threads(false), TmSmem<FMT, false>::ALLOC);
        }
    } else {
        if (gate) return cudaErrorInvalidValue;
        using R = GemmRoles<GemmCfg<FMT>::PWG>;
        e = xin ? run(gemm_kernel<FMT, true>, R::threads(true), GemmSmem<FMT, true>::ALLOC)
                : run(gemm_kernel<FMT, false>, R::threads(false), GemmSmem<FMT, false>::ALLOC);
    }
    if (e != cudaSuccess || splits == 1) return e;
    const long long count = m * (long long)n;
    long long blocks = (count + 255) / 256;
    const long long cap = (long long)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    return launch_kernel(gemm_split_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                         (const float*)part, y, count, splits);
}

// Below this many activation rows the decode GEMV kernels (eight rows at a
// time) serve the GEMM entry point.
constexpr long long GEMM_MIN_M = 9;

// Prefill on the tensor cores from GEMM_MIN_M rows: q4_K, q5_K and q6_K
// always; q2_K and q3_K when a row of blocks is a multiple of 16 bytes (nb %
// 4 == 0, resp. nb % 8 == 0: their blocks come by TMA in 16-byte windows)
// and the weights are 16-byte aligned.  Otherwise the decode GEMV runs eight
// activation rows at a time.
static bool gemm_tc_shape(int fmt, long long m, int k) {
    const int nb = k / QK;
    const bool fmt_ok = fmt == 4 || fmt == 5 || fmt == 6 || (fmt == 2 && nb % 4 == 0) || (fmt == 3 && nb % 8 == 0);
    return fmt_ok && m >= GEMM_MIN_M && m <= 0x7FFFFFFF;
}
static bool gemm_on_tensor_cores(int fmt, long long m, int k, const uint8_t* w) {
    return gemm_tc_shape(fmt, m, k) && (fmt > 3 || ((uintptr_t)w & 15u) == 0);
}

static cudaError_t gemm_tc_any(int fmt, const uint8_t* w, const uint8_t* xq, float* y, long long m, int n, int k,
                               void* ws, size_t ws_bytes, cudaStream_t stream) {
    switch (fmt) {
        case 2: return gemm_tc<2>(w, xq, y, m, n, k, ws, ws_bytes, nullptr, stream);
        case 3: return gemm_tc<3>(w, xq, y, m, n, k, ws, ws_bytes, nullptr, stream);
        case 4: return gemm_tc<4>(w, xq, y, m, n, k, ws, ws_bytes, nullptr, stream);
        case 5: return gemm_tc<5>(w, xq, y, m, n, k, ws, ws_bytes, nullptr, stream);
        default:
            // q6_K on the tensor-memory kernel when its blocks come by TMA windows (a
            // row of blocks a multiple of 16 bytes: nb % 8 == 0; 16-byte aligned weights)
            if ((k / QK) % 8 == 0 && ((uintptr_t)w & 15u) == 0)
                return gemm_tc<Q6TM>(w, xq, y, m, n, k, ws, ws_bytes, nullptr, stream);
            return gemm_tc<6>(w, xq, y, m, n, k, ws, ws_bytes, nullptr, stream);
    }
}

// Decode GEMV passes of at most eight activation rows (the GEMM entry points
// below GEMM_MIN_M rows, and q2_K / q3_K)
static cudaError_t gemm_by_gemv(int fmt, const uint8_t* w, const uint8_t* xq, float* y, long long m, int n, int k,
                                cudaStream_t stream) {
    const int nb = k / QK;
    for (long long i0 = 0; i0 < m; i0 += GEMV_MAX_M) {
        const int mm = (int)(m - i0 < GEMV_MAX_M ? m - i0 : GEMV_MAX_M);
        cudaError_t e = launch_gemv(fmt, w, xq + (size_t)i0 * nb * Q8K_BYTES, y + (size_t)i0 * n, mm, n, k, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm_ws(int fmt, const uint8_t* w, const uint8_t* xq, float* y, long long m, int n, int k,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (gemm_tc_shape(fmt, m, k) && (!ws || ws_bytes < gemm_workspace_bytes(m, k))) return cudaErrorInvalidValue;
    if (!gemm_on_tensor_cores(fmt, m, k, w)) return gemm_by_gemv(fmt, w, xq, y, m, n, k, stream);
    return gemm_tc_any(fmt, w, xq, y, m, n, k, ws, ws_bytes, stream);
}

// q4_K gate/up pair with the SwiGLU epilogue, any m.  From GEMM_MIN_M rows:
// the gate GEMM into h, the up GEMM into the front of the workspace, then one
// elementwise pass (a single launch streaming both matrices was tried and was
// slower: the epilogue of a kernel that parks g and later combines it with
// u ran out of registers).  Below: the decode GEMV pair, eight rows a launch.
static size_t pair_u_bytes(long long m, int n) { return (((size_t)m * n * 4) + 255) & ~(size_t)255; }

size_t gemm_swiglu_workspace_need(long long m, int n, int k) {
    if (!gemm_tc_shape(4, m, k)) return 0;
    return pair_u_bytes(m, n) + gemm_workspace_need_split(4, m, n, k);
}

// the least workspace the _ws pair accepts (no K split)
size_t gemm_swiglu_workspace_min(long long m, int n, int k) {
    if (!gemm_tc_shape(4, m, k)) return 0;
    return pair_u_bytes(m, n) + gemm_workspace_bytes(m, k);
}

cudaError_t launch_gemm_q4K_swiglu_ws(const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* xq, float* h,
                                      long long m, int n, int k, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (gemm_tc_shape(4, m, k)) {
        const size_t ub = pair_u_bytes(m, n);
        if (!ws || ws_bytes < ub + gemm_workspace_bytes(m, k)) return cudaErrorInvalidValue;
        float* u = static_cast<float*>(ws);
        void* gws = static_cast<uint8_t*>(ws) + ub;
        const size_t gbytes = ws_bytes - ub;
        cudaError_t e = gemm_tc<4>(w_gate, xq, h, m, n, k, gws, gbytes, nullptr, stream);
        if (e != cudaSuccess) return e;
        e = gemm_tc<4>(w_up, xq, u, m, n, k, gws, gbytes, nullptr, stream);
        if (e != cudaSuccess) return e;
        const long long count = m * (long long)n;
        long long blocks = (count + 255) / 256;
        const long long cap = (long long)num_sms() * 8;
        if (blocks > cap) blocks = cap;
        return launch_kernel(gemm_swiglu_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, h, (const float*)u,
                             count);
    }
    const int nb = k / QK;
    for (long long i0 = 0; i0 < m; i0 += GEMV_MAX_M) {
        const int mm = (int)(m - i0 < GEMV_MAX_M ? m - i0 : GEMV_MAX_M);
        GroupItem it;
        it.w = w_gate;
        it.w2 = w_up;
        it.xq = xq + (size_t)i0 * nb * Q8K_BYTES;
        it.y = h + (size_t)i0 * n;
        it.n = n;
        it.k = k;
        cudaError_t e = launch_gemv_q4K_swiglu(&it, 1, mm, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Without a workspace: the gate GEMM into h, then the up GEMM, whose
// epilogue reads each element's gate result back from h and writes
// silu(g) * u over it (same bits as the workspace form when that one does
// not split K).
cudaError_t launch_gemm_q4K_swiglu(const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* xq, float* h,
                                   long long m, int n, int k, cudaStream_t stream) {
    if (!gemm_tc_shape(4, m, k)) return launch_gemm_q4K_swiglu_ws(w_gate, w_up, xq, h, m, n, k, nullptr, 0, stream);
    cudaError_t e = gemm_tc<4>(w_gate, xq, h, m, n, k, nullptr, 0, nullptr, stream);
    if (e != cudaSuccess) return e;
    return gemm_tc<4>(w_up, xq, h, m, n, k, nullptr, 0, h, stream);
}

size_t gemm_workspace_need(int fmt, long long m, int k) {
    return gemm_tc_shape(fmt, m, k) ? gemm_workspace_bytes(m, k) : 0;
}

size_t gemm_workspace_need_split(int fmt, long long m, int n, int k) {
    if (!gemm_tc_shape(fmt, m, k)) return 0;
    return gemm_workspace_bytes(m, k) + gemm_split_bytes(m, n, gemm_splits(m, n, k / QK));
}

// Without a workspace: the tensor-core kernels widen the activation codes
// themselves and never split K; nothing is allocated.
cudaError_t launch_gemm(int fmt, const uint8_t* w, const uint8_t* xq, float* y, long long m, int n, int k,
                        cudaStream_t stream) {
    if (!gemm_on_tensor_cores(fmt, m, k, w)) return gemm_by_gemv(fmt, w, xq, y, m, n, k, stream);
    return gemm_tc_any(fmt, w, xq, y, m, n, k, nullptr, 0, stream);
}

}  // namespace plm

// ---------------------------------------------------------------------------
// Allocation-free GEMM entry through a fixed workspace: the workspace form
// of the q4_K GEMM, with its f16 activation workspace in a fixed device array
// compiled into this library.  It exists for callers
// that must not allocate device memory once they are running, for example an
// engine whose whole memory budget is claimed by its own allocator at start-up,
// or a latency-critical loop that cannot risk an allocation failing or
// waiting.  Every device that loads the library reserves the array until the
// process exits.
// ---------------------------------------------------------------------------
#include <mutex>

#include "../../include/plm.h"

namespace plm {

static __device__ __align__(256) uint8_t g_noalloc_scratch[PLM_NOALLOC_WORKSPACE_BYTES];

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and kept.
static cudaError_t noalloc_scratch_ptr(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

bool gemm_noalloc_fits(long long m, int k) {
    return gemm_workspace_need(4, m, k) <= (size_t)PLM_NOALLOC_WORKSPACE_BYTES;
}

cudaError_t launch_gemm_q4K_noalloc(const uint8_t* w, const uint8_t* xq, float* y, long long m, int n, int k,
                                    cudaStream_t stream) {
    const size_t need = gemm_workspace_need(4, m, k);
    if (need > (size_t)PLM_NOALLOC_WORKSPACE_BYTES) return cudaErrorInvalidValue;
    void* ws = nullptr;
    if (need > 0) {
        // the pre-pass rewrites all `need` bytes before the GEMM reads them,
        // so nothing left by an earlier call has to be cleared
        cudaError_t e = noalloc_scratch_ptr(&ws);
        if (e != cudaSuccess) return e;
    }
    return launch_gemm_ws(4, w, xq, y, m, n, k, ws, need, stream);
}

}  // namespace plm
