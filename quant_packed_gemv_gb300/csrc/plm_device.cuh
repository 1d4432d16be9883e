// Device-side building blocks shared by the plm kernels: block geometry,
// f16 loads, the q8_K activation staging layout in shared memory, and the
// per-lane decode + integer dot of one q4_K / q6_K block.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace plm {

// Early launch: let the next kernel of the stream be scheduled, and wait for
// the kernels before this one (and their memory) before touching memory
// they write.  Both are no-ops for a kernel launched in plain stream order.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

constexpr int QK = 256;          // weights (or activations) per block
constexpr int Q2K_BYTES = 84;    // scales[16], qs[64], f16 d, f16 dmin
constexpr int Q3K_BYTES = 110;   // hmask[32], qs[64], scales[12], f16 d
constexpr int Q4K_BYTES = 144;   // f16 d, f16 dmin, scales[12], qs[128]
constexpr int Q5K_BYTES = 176;   // f16 d, f16 dmin, scales[12], qh[32], qs[128]
constexpr int Q6K_BYTES = 210;   // ql[128], qh[64], scales[16], f16 d
constexpr int Q8K_BYTES = 292;   // f32 d, qs[256], bsums[16]
constexpr int GEMV_MAX_M = 8;

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
    __half_raw r;
    r.x = (unsigned short)(bits16 & 0xFFFFu);
    return __half2float(__half(r));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ int dp4a(int a, int b, int c) { return __dp4a(a, b, c); }

// ---------------------------------------------------------------------------
// q8_K activations staged in shared memory, re-laid out for aligned access:
//   q8  : int8  [M*nb][256]     16-byte chunks XOR-swizzled per block
//   bs  : int16 [M*nb][16]      (32 bytes per block, 16-byte aligned)
//   dy  : float [M*nb]
// Chunk c (bytes 16c..16c+15) of staged block blk sits at chunk slot
// act_swizzle<FMT>(c, blk).  The swizzle spreads the four lanes of a block,
// and the two blocks of an 8-lane phase, over distinct bank groups for the
// access pattern of each format's lane decode.
// ---------------------------------------------------------------------------
struct ActSmem {
    int8_t* q8;
    int16_t* bs;
    float* dy;
};

template <int FMT>
__host__ __device__ __forceinline__ int act_swizzle(int c, int blk) {
    const int x = FMT == 4 ? (blk & 1) : ((blk & 1) << 2);
    return c ^ ((c >> 3) << 1) ^ x;
}

template <int FMT>
__device__ __forceinline__ const int4* act_chunk(const ActSmem& a, int blk, int c) {
    return reinterpret_cast<const int4*>(a.q8 + (size_t)blk * QK + 16 * act_swizzle<FMT>(c, blk));
}

__host__ __device__ inline size_t act_smem_bytes(int m, int nb) {
    return (size_t)m * nb * (QK + 32 + 4);
}

__device__ __forceinline__ ActSmem act_smem_carve(uint8_t* base, int m, int nb) {
    ActSmem a;
    a.q8 = reinterpret_cast<int8_t*>(base);
    a.bs = reinterpret_cast<int16_t*>(base + (size_t)m * nb * QK);
    a.dy = reinterpret_cast<float*>(base + (size_t)m * nb * (QK + 32));
    return a;
}

// Copies m*nb q8_K blocks (4-byte aligned) into the staged layout. All
// threads of the CTA take part; the caller synchronizes afterwards.
template <int FMT>
__device__ __forceinline__ void act_smem_fill(const ActSmem& a, const uint8_t* __restrict__ xq,
                                              int m, int nb) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(xq);
    const int words_per_block = Q8K_BYTES / 4;  // 73
    const int total = m * nb * words_per_block;
    uint32_t* q8w = reinterpret_cast<uint32_t*>(a.q8);
    uint32_t* bsw = reinterpret_cast<uint32_t*>(a.bs);
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int blk = idx / words_per_block;
        const int wd = idx - blk * words_per_block;
        const uint32_t v = __ldg(src + idx);
        if (wd == 0) {
            a.dy[blk] = __uint_as_float(v);
        } else if (wd <= 64) {
            const int w = wd - 1;
            q8w[blk * 64 + 4 * act_swizzle<FMT>(w >> 2, blk) + (w & 3)] = v;
        } else {
            bsw[blk * 8 + (wd - 65)] = v;
        }
    }
}

// ---------------------------------------------------------------------------
// Mixed-sign integer dot products used by the block decoders.
// ---------------------------------------------------------------------------

// Mixed-sign 4-way byte dot: unsigned bytes of a times signed bytes of b.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two-way dot: signed 16-bit halves of a times unsigned bytes 0, 1 of b.
__device__ __forceinline__ int dp2a_lo_su(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------------------
// q6_K, one block handled by 4 lanes.  Lane t: half h = t/2, p = t%2 owns
// l in [16p, 16p+16) of every quarter qq of half h, i.e. the weights
//   128h + 32qq + 16p + [0,16)  =  the whole 16-group G = 8h + 2qq + p.
// Quarter qq takes its low 4 bits from ql[64h + 32(qq&1) + l] (low nibble for
// qq < 2, high nibble otherwise) and its top 2 bits from bits 2qq..2qq+1 of
// qh[32h + l].
// ---------------------------------------------------------------------------
struct Q6KLane {
    float d;
    int sc[4];               // scale of group 8h + 2qq + p
    uint32_t code[4][4];     // 16 six-bit codes per quarter, one per byte
};

// A = ql[64h+16p .. +16], B = ql[64h+32+16p .. +16], H = qh[32h+16p .. +16],
// S = scales[8h .. 8h+8] (i8), dbits = f16 d
__device__ __forceinline__ Q6KLane q6K_lane_decode(uint4 A, uint4 B, uint4 H, uint2 S, uint32_t dbits, int p) {
    Q6KLane L;
    L.d = half_bits_to_float(dbits);
    const uint32_t a[4] = {A.x, A.y, A.z, A.w};
    const uint32_t bq[4] = {B.x, B.y, B.z, B.w};
    const uint32_t hh[4] = {H.x, H.y, H.z, H.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        L.code[0][i] = (a[i] & 0x0F0F0F0Fu) | ((hh[i] << 4) & 0x30303030u);
        L.code[1][i] = (bq[i] & 0x0F0F0F0Fu) | ((hh[i] << 2) & 0x30303030u);
        L.code[2][i] = ((a[i] >> 4) & 0x0F0F0F0Fu) | (hh[i] & 0x30303030u);
        L.code[3][i] = ((bq[i] >> 4) & 0x0F0F0F0Fu) | ((hh[i] >> 2) & 0x30303030u);
    }
    const uint32_t sw[2] = {S.x, S.y};
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const int byte = 2 * qq + p;
        L.sc[qq] = (int)(int8_t)((sw[byte >> 2] >> (8 * (byte & 3))) & 0xFFu);
    }
    return L;
}

// Raw dot of quarter qq's 16 codes (q6 in 0..63) with the activation codes
// x8 at 128h + 32qq + 16p.  The exact group dot is raw - 32*bsum_G.
__device__ __forceinline__ int q6K_lane_raw(const Q6KLane& L, int qq, int4 x8) {
    int r = dp4a((int)L.code[qq][0], x8.x, 0);
    r = dp4a((int)L.code[qq][1], x8.y, r);
    r = dp4a((int)L.code[qq][2], x8.z, r);
    return dp4a((int)L.code[qq][3], x8.w, r);
}

// Reads 16 bytes at an even (2-byte aligned) shared-memory offset using
// aligned 4-byte loads and funnel shifts.
__device__ __forceinline__ uint4 lds16_align2(const uint8_t* base, int off) {
    const int a = off & ~3;
    const uint32_t* p = reinterpret_cast<const uint32_t*>(base + a);
    const uint32_t w0 = p[0], w1 = p[1], w2 = p[2], w3 = p[3], w4 = p[4];
    const int sh = (off & 3) * 8;
    return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                      __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

// Reads 8 bytes at an even (2-byte aligned) shared-memory offset using
// aligned 4-byte loads and a funnel shift.
__device__ __forceinline__ uint2 lds8_align2(const uint8_t* base, int off) {
    const int a = off & ~3;
    const uint32_t* p = reinterpret_cast<const uint32_t*>(base + a);
    const uint32_t w0 = p[0], w1 = p[1], w2 = p[2];
    const int sh = (off & 3) * 8;
    uint2 r;
    r.x = __funnelshift_r(w0, w1, sh);
    r.y = __funnelshift_r(w1, w2, sh);
    return r;
}

// q8_K quantization of one 256-value chunk by one warp; lane L holds values
// 8L .. 8L+7 in v[].  Signed amax with the first occurrence winning (the
// index is carried through the reduction), iscale = -128/max and
// d = 1/iscale as IEEE f32 divisions, codes min(127, rne(iscale * x)) from a
// single rounded multiply; an all-zero chunk gives d = 0 and zero codes.
// Writes the lane's eight codes and returns d.
__device__ __forceinline__ float q8K_quantize_warp(const float v[8], int lane, int q[8]) {
    float amax = 0.0f;
    int idx = 0x7FFFFFFF;
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float av = fabsf(v[i]);
        if (av > amax) { amax = av; mx = v[i]; idx = 8 * lane + i; }
    }
    // larger magnitude wins; on equal magnitude the smaller index wins
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oa = __shfl_xor_sync(0xFFFFFFFFu, amax, o);
        const float om = __shfl_xor_sync(0xFFFFFFFFu, mx, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
        if (oa > amax || (oa == amax && oi < idx)) { amax = oa; mx = om; idx = oi; }
    }
    if (amax == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = 0;
        return 0.0f;
    }
    const float iscale = __fdiv_rn(-128.0f, mx);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = min(127, __float2int_rn(__fmul_rn(iscale, v[i])));
    return __fdiv_rn(1.0f, iscale);
}

__device__ __forceinline__ void pack_codes8(const int q[8], uint32_t& w0, uint32_t& w1) {
    w0 = 0;
    w1 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w0 |= (uint32_t)(q[i] & 0xFF) << (8 * i);
        w1 |= (uint32_t)(q[4 + i] & 0xFF) << (8 * i);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace plm

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA, 1-D) helpers.  Every wait is bounded: a wait that
// runs out sets a device fault word and returns false, and the caller stops
// issuing work.
// ---------------------------------------------------------------------------
namespace plm {

constexpr unsigned WAIT_LIMIT = 1u << 16;   // try_wait rounds before giving up (each up to SUSPEND_NS)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// Returns true once the phase with the given parity has completed, false if
// `limit` rounds (WAIT_LIMIT unless given) pass first.  Each round lets the
// hardware suspend the warp for up to SUSPEND_NS (it resumes as soon as the
// phase completes), so waiting warps do not spin on the issue slots.
constexpr unsigned SUSPEND_NS = 20000;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned limit = WAIT_LIMIT) {
    const uint32_t a = smem_u32(bar);
    for (unsigned it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(a), "r"(parity), "r"(SUSPEND_NS) : "memory");
        if (done) return true;
    }
    return false;
}

// Bulk copy global -> shared (this CTA), completion counted on `bar`.
// src and dst 16-byte aligned, bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

}  // namespace plm
