// Device-side building blocks shared by the plm kernels: block geometry,
// f16 loads, the q8_K activation staging layout in shared memory, and the
// per-lane decode + integer dot of one q4_K / q6_K block.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace plm {

constexpr int QK = 256;          // weights (or activations) per block
constexpr int Q4K_BYTES = 144;   // f16 d, f16 dmin, scales[12], qs[128]
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
//   q8  : int8  [M][k]          (16-byte aligned rows)
//   dy  : float [M][nb]
//   bs  : int16 [M][nb][16]
// ---------------------------------------------------------------------------
struct ActSmem {
    int8_t* q8;
    float* dy;
    int16_t* bs;
};

__host__ __device__ inline size_t act_smem_bytes(int m, int nb) {
    return (size_t)m * nb * QK + (size_t)m * nb * 4 + (size_t)m * nb * 32;
}

__device__ __forceinline__ ActSmem act_smem_carve(uint8_t* base, int m, int nb) {
    ActSmem a;
    a.q8 = reinterpret_cast<int8_t*>(base);
    a.dy = reinterpret_cast<float*>(base + (size_t)m * nb * QK);
    a.bs = reinterpret_cast<int16_t*>(base + (size_t)m * nb * QK + (size_t)m * nb * 4);
    return a;
}

// Copies m*nb q8_K blocks (4-byte aligned) into the staged layout. All
// threads of the CTA take part; the caller synchronizes afterwards.
__device__ __forceinline__ void act_smem_fill(const ActSmem& a, const uint8_t* __restrict__ xq,
                                              int m, int nb) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(xq);
    const int words_per_block = Q8K_BYTES / 4;  // 73
    const int total = m * nb * words_per_block;
    uint32_t* q8w = reinterpret_cast<uint32_t*>(a.q8);
    uint32_t* bsw = reinterpret_cast<uint32_t*>(a.bs);
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        int blk = idx / words_per_block;
        int wd = idx - blk * words_per_block;
        uint32_t v = __ldg(src + idx);
        if (wd == 0) {
            a.dy[blk] = __uint_as_float(v);
        } else if (wd <= 64) {
            q8w[blk * 64 + (wd - 1)] = v;
        } else {
            bsw[blk * 8 + (wd - 65)] = v;
        }
    }
}

// ---------------------------------------------------------------------------
// q4_K, one block handled by 8 lanes.  Lane t (0..7) owns qs bytes
// [16t, 16t+16): chunk c = t/2, half p = t%2, i.e. weights
//   64c + 16p + [0,16)       in the low nibbles  (sub-block 2c)
//   64c + 32 + 16p + [0,16)  in the high nibbles (sub-block 2c+1)
// ---------------------------------------------------------------------------
struct Q4KLane {
    float d, dmin;
    int sc_lo, sc_hi, m_lo, m_hi;
    uint32_t lo[4], hi[4];  // 16 four-bit codes each, one per byte
};

// hdr: bytes 0..15 of the block (d, dmin, scales[12]); qv: qs[16t..16t+15]
__device__ __forceinline__ Q4KLane q4K_lane_decode(uint4 hdr, uint4 qv, int t) {
    Q4KLane L;
    L.d = half_bits_to_float(hdr.x);
    L.dmin = half_bits_to_float(hdr.x >> 16);
    const int c = t >> 1;
    uint32_t scw, mw;
    if (c < 2) {   // pairs 0..3: low six bits of scale bytes 0..3 / 4..7
        scw = hdr.y & 0x3F3F3F3Fu;
        mw = hdr.z & 0x3F3F3F3Fu;
    } else {       // pairs 4..7: nibbles of bytes 8..11 + top bits of bytes 0..7
        scw = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
        mw = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    }
    const int sh = 16 * (c & 1);
    L.sc_lo = (scw >> sh) & 0xFF;
    L.sc_hi = (scw >> (sh + 8)) & 0xFF;
    L.m_lo = (mw >> sh) & 0xFF;
    L.m_hi = (mw >> (sh + 8)) & 0xFF;
    const uint32_t q[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        L.lo[u] = q[u] & 0x0F0F0F0Fu;
        L.hi[u] = (q[u] >> 4) & 0x0F0F0F0Fu;
    }
    return L;
}

// Integer dots of the lane's 16 low-nibble and 16 high-nibble weights against
// the matching activation codes (q8lo at weight 64c+16p, q8hi at 64c+32+16p).
__device__ __forceinline__ void q4K_lane_dots(const Q4KLane& L, int4 q8lo, int4 q8hi,
                                              int& dlo, int& dhi) {
    dlo = dp4a((int)L.lo[0], q8lo.x, 0);
    dlo = dp4a((int)L.lo[1], q8lo.y, dlo);
    dlo = dp4a((int)L.lo[2], q8lo.z, dlo);
    dlo = dp4a((int)L.lo[3], q8lo.w, dlo);
    dhi = dp4a((int)L.hi[0], q8hi.x, 0);
    dhi = dp4a((int)L.hi[1], q8hi.y, dhi);
    dhi = dp4a((int)L.hi[2], q8hi.z, dhi);
    dhi = dp4a((int)L.hi[3], q8hi.w, dhi);
}

// ---------------------------------------------------------------------------
// q6_K, one block handled by 8 lanes.  Lane t: half h = t/4, u = t%4 owns
// l in [8u, 8u+8) of every quarter of half h, i.e. the weights
//   128h + 32*qq + 8u + [0,8),  qq = 0..3
// Quarter qq takes its low 4 bits from ql[64h + 32*(qq&1) + l] (low nibble
// for qq < 2, high nibble otherwise) and its top 2 bits from bits 2qq..2qq+1
// of qh[32h + l].  Its scale / 16-group is 8h + 2qq + u/2.
// ---------------------------------------------------------------------------
struct Q6KLane {
    float d;
    int sc[4];          // scale of quarter qq's group
    uint32_t code[4][2];  // 8 six-bit codes per quarter, one per byte
};

// qlA = ql[64h+8u .. +8], qlB = ql[64h+32+8u .. +8], qhv = qh[32h+8u .. +8],
// scw = scales[8h .. 8h+8] (i8), dbits = f16 d
__device__ __forceinline__ Q6KLane q6K_lane_decode(uint2 qlA, uint2 qlB, uint2 qhv, uint2 scw,
                                                   uint32_t dbits, int u) {
    Q6KLane L;
    L.d = half_bits_to_float(dbits);
    const uint32_t sca[2] = {scw.x, scw.y};
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const int byte = 2 * qq + (u >> 1);   // index into scales[8h..8h+8)
        L.sc[qq] = (int)(int8_t)((sca[byte >> 2] >> (8 * (byte & 3))) & 0xFF);
        const uint2 src = (qq & 1) ? qlB : qlA;
        const int nsh = (qq & 2) ? 4 : 0;
        const int hsh = 2 * qq;
        L.code[qq][0] = ((src.x >> nsh) & 0x0F0F0F0Fu) | (((qhv.x >> hsh) & 0x03030303u) << 4);
        L.code[qq][1] = ((src.y >> nsh) & 0x0F0F0F0Fu) | (((qhv.y >> hsh) & 0x03030303u) << 4);
    }
    return L;
}

// Raw (unshifted) dots: sum over the lane's 8 weights of quarter qq of q6*q8,
// q6 in 0..63.  The -32 offset is applied with the q8_K bsums:
//   dot_g = raw(lane u even) + raw(lane u odd) - 32*bsum_g.
__device__ __forceinline__ int q6K_lane_raw(const Q6KLane& L, int qq, int2 q8v) {
    int r = dp4a((int)L.code[qq][0], q8v.x, 0);
    return dp4a((int)L.code[qq][1], q8v.y, r);
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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace plm
