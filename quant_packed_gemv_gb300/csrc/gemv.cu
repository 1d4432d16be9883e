// Decode GEMV for m = 1..8 activation rows over packed q4_K / q6_K weights
// (PocketLLM "What it runs": K-quant weights decoded inside the kernel,
// never widened; the weight stream is read once for all m activation rows,
// as the pages' 8-row activation tile does on the CPU).
//
// Layout of the work: a CTA of 8 warps stages all m rows of q8_K activations
// in shared memory once, then each warp takes whole weight rows.  Inside a
// warp, 8 lanes share one 256-weight block: 4 blocks of a row per step.
// Per block and activation row every lane forms integer dots with dp4a,
// folds the sub-block scales in int32, and adds one f32 term
// dy * (d*isum - dmin*msum); the warp reduces with shuffles at the row end.
// The per-lane f32 sequence is pinned with explicit _rn intrinsics, so the
// result for activation row i is the same for every m.
//
// q6_K blocks are 210 bytes, so a block is only 2-byte aligned in memory.
// Each warp stages 8 blocks of its row at a time through shared memory with
// aligned 16-byte loads and reads fields back with funnel shifts.
//
// With SUBDOTS the same kernel writes the integer sub-block dots instead of
// the f32 result (verification export).
#include "plm_device.cuh"
#include "plm_internal.h"

namespace plm {

constexpr int GEMV_THREADS = 256;
constexpr int GEMV_WARPS = GEMV_THREADS / 32;
constexpr int Q6K_STAGE_BLOCKS = 8;
constexpr int Q6K_STAGE_BYTES = 1728;  // 8*210 + alignment slack, multiple of 16

__device__ __forceinline__ uint4 ldg_v4(const uint8_t* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

template <int M, bool SUBDOTS>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_q4K_kernel(const uint8_t* __restrict__ w,
                                                                const uint8_t* __restrict__ xq,
                                                                float* __restrict__ y,
                                                                int32_t* __restrict__ sub,
                                                                int n, int nb) {
    extern __shared__ __align__(16) uint8_t smem[];
    const ActSmem a = act_smem_carve(smem, M, nb);
    act_smem_fill(a, xq, M, nb);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 3, t = lane & 7, c = t >> 1, p = t & 1;
    const int lo_off = 64 * c + 16 * p, hi_off = lo_off + 32;
    const int g_lo = 4 * c + p, g_hi = g_lo + 2;

    for (int r = blockIdx.x * GEMV_WARPS + warp; r < n; r += gridDim.x * GEMV_WARPS) {
        const uint8_t* row = w + (size_t)r * nb * Q4K_BYTES;
        float acc[M];
#pragma unroll
        for (int i = 0; i < M; ++i) acc[i] = 0.0f;
#pragma unroll 2
        for (int b = g; b < nb; b += 4) {
            const uint8_t* blk = row + (size_t)b * Q4K_BYTES;
            const uint4 hdr = ldg_v4(blk);
            const uint4 qv = ldg_v4(blk + 16 + 16 * t);
            const Q4KLane L = q4K_lane_decode(hdr, qv, t);
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const int8_t* q8 = a.q8 + ((size_t)i * nb + b) * QK;
                const int4 q8lo = *reinterpret_cast<const int4*>(q8 + lo_off);
                const int4 q8hi = *reinterpret_cast<const int4*>(q8 + hi_off);
                int dlo, dhi;
                q4K_lane_dots(L, q8lo, q8hi, dlo, dhi);
                if constexpr (SUBDOTS) {
                    const unsigned gmask = 0xFFu << (8 * g);   // the 8 lanes of this block
                    dlo += __shfl_xor_sync(gmask, dlo, 1);
                    dhi += __shfl_xor_sync(gmask, dhi, 1);
                    if (p == 0) {
                        int32_t* o = sub + (((size_t)i * n + r) * nb + b) * 8;
                        o[2 * c] = dlo;
                        o[2 * c + 1] = dhi;
                    }
                } else {
                    const int isum = L.sc_lo * dlo + L.sc_hi * dhi;
                    const int16_t* bs = a.bs + ((size_t)i * nb + b) * 16;
                    const int msum = L.m_lo * (int)bs[g_lo] + L.m_hi * (int)bs[g_hi];
                    const float tt = __fmaf_rn(L.d, (float)isum, -__fmul_rn(L.dmin, (float)msum));
                    acc[i] = __fmaf_rn(a.dy[i * nb + b], tt, acc[i]);
                }
            }
        }
        if constexpr (!SUBDOTS) {
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const float s = warp_sum(acc[i]);
                if (lane == 0) y[(size_t)i * n + r] = s;
            }
        }
    }
}

template <int M, bool SUBDOTS>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_q6K_kernel(const uint8_t* __restrict__ w,
                                                                const uint8_t* __restrict__ xq,
                                                                float* __restrict__ y,
                                                                int32_t* __restrict__ sub,
                                                                int n, int nb, long long wbytes) {
    extern __shared__ __align__(16) uint8_t smem[];
    const ActSmem a = act_smem_carve(smem, M, nb);
    const size_t act_bytes = (act_smem_bytes(M, nb) + 15) & ~(size_t)15;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t* stage = smem + act_bytes + (size_t)warp * Q6K_STAGE_BYTES;
    act_smem_fill(a, xq, M, nb);
    __syncthreads();

    const int g = lane >> 3, t = lane & 7, h = t >> 2, u = t & 3;

    for (int r = blockIdx.x * GEMV_WARPS + warp; r < n; r += gridDim.x * GEMV_WARPS) {
        const long long row_off = (long long)r * nb * Q6K_BYTES;
        float acc[M];
#pragma unroll
        for (int i = 0; i < M; ++i) acc[i] = 0.0f;
        for (int b0 = 0; b0 < nb; b0 += Q6K_STAGE_BLOCKS) {
            const int cnt = min(Q6K_STAGE_BLOCKS, nb - b0);
            const long long S = row_off + (long long)Q6K_BYTES * b0;
            const long long A0 = S & ~15LL;
            const int delta = (int)(S - A0);
            const int npieces = (delta + Q6K_BYTES * cnt + 15) >> 4;
            __syncwarp();
            for (int q = lane; q < npieces; q += 32) {
                const long long gaddr = A0 + 16LL * q;
                uint4 v;
                if (gaddr + 16 <= wbytes) {
                    v = ldg_v4(w + gaddr);
                } else {   // last piece of the matrix: never read past its end
                    uint32_t tmp[4] = {0u, 0u, 0u, 0u};
                    for (int j = 0; j < 16 && gaddr + j < wbytes; ++j)
                        tmp[j >> 2] |= (uint32_t)w[gaddr + j] << (8 * (j & 3));
                    v = make_uint4(tmp[0], tmp[1], tmp[2], tmp[3]);
                }
                *reinterpret_cast<uint4*>(stage + 16 * q) = v;
            }
            __syncwarp();
            for (int j = g; j < cnt; j += 4) {
                const int base = delta + Q6K_BYTES * j;
                const uint2 qlA = lds8_align2(stage, base + 64 * h + 8 * u);
                const uint2 qlB = lds8_align2(stage, base + 64 * h + 32 + 8 * u);
                const uint2 qhv = lds8_align2(stage, base + 128 + 32 * h + 8 * u);
                const uint2 scw = lds8_align2(stage, base + 192 + 8 * h);
                const uint32_t dbits = *reinterpret_cast<const uint16_t*>(stage + base + 208);
                const Q6KLane L = q6K_lane_decode(qlA, qlB, qhv, scw, dbits, u);
                const int b = b0 + j;
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    const int8_t* q8 = a.q8 + ((size_t)i * nb + b) * QK;
                    const int16_t* bs = a.bs + ((size_t)i * nb + b) * 16;
                    int isum = 0;
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const int2 q8v = *reinterpret_cast<const int2*>(q8 + 128 * h + 32 * qq + 8 * u);
                        const int raw = q6K_lane_raw(L, qq, q8v);
                        const int G = 8 * h + 2 * qq + (u >> 1);
                        if constexpr (SUBDOTS) {
                            const unsigned gmask = 0xFFu << (8 * g);
                            const int both = raw + __shfl_xor_sync(gmask, raw, 1);
                            if ((u & 1) == 0)
                                sub[(((size_t)i * n + r) * nb + b) * 16 + G] = both - 32 * (int)bs[G];
                        } else {
                            const int corr = (u & 1) ? 0 : 32 * (int)bs[G];
                            isum += L.sc[qq] * (raw - corr);
                        }
                    }
                    if constexpr (!SUBDOTS)
                        acc[i] = __fmaf_rn(__fmul_rn(L.d, a.dy[i * nb + b]), (float)isum, acc[i]);
                }
            }
        }
        if constexpr (!SUBDOTS) {
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const float s = warp_sum(acc[i]);
                if (lane == 0) y[(size_t)i * n + r] = s;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host launch
// ---------------------------------------------------------------------------
static size_t gemv_smem_bytes(int fmt, int m, int nb) {
    size_t s = (act_smem_bytes(m, nb) + 15) & ~(size_t)15;
    if (fmt == 6) s += (size_t)GEMV_WARPS * Q6K_STAGE_BYTES;
    return s;
}

template <int M, bool SUB>
static cudaError_t launch_one(int fmt, const uint8_t* w, const uint8_t* xq, float* y, int32_t* sub,
                              int n, int nb, cudaStream_t stream) {
    const size_t smem = gemv_smem_bytes(fmt, M, nb);
    const void* fn = fmt == 4 ? (const void*)gemv_q4K_kernel<M, SUB> : (const void*)gemv_q6K_kernel<M, SUB>;
    cudaError_t e;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, GEMV_THREADS, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = ((long long)n + GEMV_WARPS - 1) / GEMV_WARPS;
    const long long cap = (long long)num_sms() * per_sm;
    if (grid > cap) grid = cap;
    if (fmt == 4) {
        gemv_q4K_kernel<M, SUB><<<(unsigned)grid, GEMV_THREADS, smem, stream>>>(w, xq, y, sub, n, nb);
    } else {
        const long long wbytes = (long long)n * nb * Q6K_BYTES;
        gemv_q6K_kernel<M, SUB><<<(unsigned)grid, GEMV_THREADS, smem, stream>>>(w, xq, y, sub, n, nb, wbytes);
    }
    return cudaGetLastError();
}

template <bool SUB>
static cudaError_t dispatch_m(int fmt, const uint8_t* w, const uint8_t* xq, float* y, int32_t* sub,
                              int m, int n, int nb, cudaStream_t stream) {
    switch (m) {
        case 1: return launch_one<1, SUB>(fmt, w, xq, y, sub, n, nb, stream);
        case 2: return launch_one<2, SUB>(fmt, w, xq, y, sub, n, nb, stream);
        case 3: return launch_one<3, SUB>(fmt, w, xq, y, sub, n, nb, stream);
        case 4: return launch_one<4, SUB>(fmt, w, xq, y, sub, n, nb, stream);
        case 5: return launch_one<5, SUB>(fmt, w, xq, y, sub, n, nb, stream);
        case 6: return launch_one<6, SUB>(fmt, w, xq, y, sub, n, nb, stream);
        case 7: return launch_one<7, SUB>(fmt, w, xq, y, sub, n, nb, stream);
        case 8: return launch_one<8, SUB>(fmt, w, xq, y, sub, n, nb, stream);
        default: return cudaErrorInvalidValue;
    }
}

// The staged activations must fit the shared memory of one CTA; when m*k is
// too large, the activation rows are taken in smaller groups (each group
// re-reads W).  Row i of every group gives the same result as in one pass.
static int gemv_rows_per_pass(int fmt, int m, int nb) {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    int rows = m;
    while (rows > 1 && gemv_smem_bytes(fmt, rows, nb) > (size_t)optin) --rows;
    return rows;
}

static cudaError_t run(int fmt, const uint8_t* w, const uint8_t* xq, float* y, int32_t* sub,
                       int m, int n, int k, cudaStream_t stream, bool subdots) {
    const int nb = k / QK;
    const int step = gemv_rows_per_pass(fmt, m, nb);
    for (int i0 = 0; i0 < m; i0 += step) {
        const int mm = min(step, m - i0);
        const uint8_t* xqi = xq + (size_t)i0 * nb * Q8K_BYTES;
        cudaError_t e;
        if (subdots) {
            const int per = fmt == 4 ? 8 : 16;
            e = dispatch_m<true>(fmt, w, xqi, nullptr, sub + (size_t)i0 * n * nb * per, mm, n, nb, stream);
        } else {
            e = dispatch_m<false>(fmt, w, xqi, y + (size_t)i0 * n, nullptr, mm, n, nb, stream);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool gemv_supported(int fmt, int k) {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return gemv_smem_bytes(fmt, 1, k / QK) <= (size_t)optin;
}

cudaError_t launch_gemv(int fmt, const uint8_t* w, const uint8_t* xq, float* y,
                        int m, int n, int k, cudaStream_t stream) {
    return run(fmt, w, xq, y, nullptr, m, n, k, stream, false);
}

cudaError_t launch_subdots(int fmt, const uint8_t* w, const uint8_t* xq, int32_t* out,
                           int m, int n, int k, cudaStream_t stream) {
    return run(fmt, w, xq, nullptr, out, m, n, k, stream, true);
}

}  // namespace plm
