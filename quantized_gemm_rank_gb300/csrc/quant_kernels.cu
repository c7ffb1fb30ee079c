// quant_kernels.cu -- the memory-bound steps of AlltoAllQuantMatmul
// ("aclnnAlltoAllQuantMatmul", 功能说明 / 计算公式):
//   * the per-token dynamic quant prologue of the dynamic-quant scenario,
//     reading the rank's received chunks through the permute(1,0,2) index
//     (permuted[t, r*h + j] = chunk_r[t, j]) without materialising the
//     permuted bf16/fp16 matrix;
//   * the exact int8 -> fp16 widening of the int8 operands that the tensor
//     cores consume (sm_103a has no integer tcgen05 MMA);
//   * the optional alltoAllOut output (commOut, the rank_size received blocks
//     stacked as (rank_size, bs_local, h) in x1's dtype), stored from the same
//     registers that read the chunks.
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mc2 {

namespace {

template <bool kBF16>
__device__ __forceinline__ float to_f32(uint16_t v) {
    if constexpr (kBF16) {
        return __uint_as_float(static_cast<uint32_t>(v) << 16);
    } else {
        return __half2float(__ushort_as_half(v));
    }
}

// Four int8 values (one 32-bit word) -> four exact fp16 values, without a
// conversion instruction: flipping the sign bits gives x + 128 in [0, 255];
// as the low mantissa byte under the fp16 exponent of 1024 (0x64) that is
// the half 1024 + x + 128, and subtracting 1152 (0x6480) leaves x exactly.
__device__ __forceinline__ uint2 i8x4_to_f16x4(uint32_t w) {
    const uint32_t b = w ^ 0x80808080u;
    const uint32_t lo = __byte_perm(b, 0x64646464u, 0x4140u);   // halves 1024 + b0, 1024 + b1
    const uint32_t hi = __byte_perm(b, 0x64646464u, 0x4342u);   // halves 1024 + b2, 1024 + b3
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 l = __hsub2(*reinterpret_cast<const __half2 *>(&lo), bias);
    const __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&hi), bias);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&l), *reinterpret_cast<const uint32_t *>(&h));
}

// 16 int8 values -> 16 fp16 values (two 16-byte vectors).
__device__ __forceinline__ void i8x16_to_f16x16(const int4 &v, uint4 (&o)[2]) {
    const uint2 a = i8x4_to_f16x4(static_cast<uint32_t>(v.x));
    const uint2 b = i8x4_to_f16x4(static_cast<uint32_t>(v.y));
    const uint2 c = i8x4_to_f16x4(static_cast<uint32_t>(v.z));
    const uint2 d = i8x4_to_f16x4(static_cast<uint32_t>(v.w));
    o[0] = make_uint4(a.x, a.y, b.x, b.y);
    o[1] = make_uint4(c.x, c.y, d.x, d.y);
}

__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    const float r = red[0];
    __syncthreads();
    return r;
}

// q = clamp(rne(y / scale), -127, 127); a zero scale (all-zero row) gives 0.
__device__ __forceinline__ int quant1(float y, float scale) {
    if (scale == 0.0f) return 0;
    const int q = __float2int_rn(__fdiv_rn(y, scale));
    return max(-127, min(127, q));
}

// One CTA per permuted row t.  Pass 1: y = x * smooth (fp32), row absmax.
// scale = absmax / 127 (IEEE division).  Pass 2 (row re-read from L1/L2):
// q, written as exact fp16 (GEMM operand) and optionally as int8.
template <bool kBF16>
__global__ void __launch_bounds__(256) quant_pertoken_kernel(const __grid_constant__ ChunkPtrs chunks, int h, int64_t bs_local, int rank_size,
                                                             const uint16_t *__restrict__ smooth,
                                                             __half *__restrict__ qh, int8_t *__restrict__ q_out,
                                                             float *__restrict__ scale_out,
                                                             uint16_t *__restrict__ comm_out) {
    ptx::allow_dependent_launch();
    __shared__ float red[32];
    const int K = rank_size * h;
    const bool vec = (h % 8) == 0;
    for (int64_t t = blockIdx.x; t < bs_local; t += gridDim.x) {
        float amax = 0.0f;
        if (vec) {
            for (int v = threadIdx.x; v < K / 8; v += blockDim.x) {
                const int c = v * 8;
                const int r = c / h;
                const int j = c - r * h;
                const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(
                    static_cast<const uint16_t *>(chunks.p[r]) + t * h + j));
                if (comm_out) *reinterpret_cast<uint4 *>(comm_out + (r * bs_local + t) * h + j) = xv;
                uint4 sv = make_uint4(0, 0, 0, 0);
                if (smooth) sv = __ldg(reinterpret_cast<const uint4 *>(smooth + c));
                const uint16_t *xe = reinterpret_cast<const uint16_t *>(&xv);
                const uint16_t *se = reinterpret_cast<const uint16_t *>(&sv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float y = smooth ? __fmul_rn(to_f32<kBF16>(xe[e]), to_f32<kBF16>(se[e]))
                                           : to_f32<kBF16>(xe[e]);
                    amax = fmaxf(amax, fabsf(y));
                }
            }
        } else {
            for (int c = threadIdx.x; c < K; c += blockDim.x) {
                const int r = c / h;
                const int j = c - r * h;
                const uint16_t xr = static_cast<const uint16_t *>(chunks.p[r])[t * h + j];
                if (comm_out) comm_out[(r * bs_local + t) * h + j] = xr;
                const float x = to_f32<kBF16>(xr);
                const float y = smooth ? __fmul_rn(x, to_f32<kBF16>(smooth[c])) : x;
                amax = fmaxf(amax, fabsf(y));
            }
        }
        amax = block_max(amax, red);
        const float scale = __fdiv_rn(amax, 127.0f);
        if (threadIdx.x == 0) scale_out[t] = scale;
        __half *qrow = qh + t * K;
        int8_t *orow = q_out ? q_out + t * K : nullptr;
        if (vec) {
            for (int v = threadIdx.x; v < K / 8; v += blockDim.x) {
                const int c = v * 8;
                const int r = c / h;
                const int j = c - r * h;
                const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(
                    static_cast<const uint16_t *>(chunks.p[r]) + t * h + j));
                uint4 sv = make_uint4(0, 0, 0, 0);
                if (smooth) sv = __ldg(reinterpret_cast<const uint4 *>(smooth + c));
                const uint16_t *xe = reinterpret_cast<const uint16_t *>(&xv);
                const uint16_t *se = reinterpret_cast<const uint16_t *>(&sv);
                uint4 hv;
                uint16_t *he = reinterpret_cast<uint16_t *>(&hv);
                uint2 iv;
                int8_t *ie = reinterpret_cast<int8_t *>(&iv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float y = smooth ? __fmul_rn(to_f32<kBF16>(xe[e]), to_f32<kBF16>(se[e]))
                                           : to_f32<kBF16>(xe[e]);
                    const int q = quant1(y, scale);
                    he[e] = __half_as_ushort(__int2half_rn(q));
                    ie[e] = static_cast<int8_t>(q);
                }
                *reinterpret_cast<uint4 *>(qrow + c) = hv;
                if (orow) *reinterpret_cast<uint2 *>(orow + c) = iv;
            }
        } else {
            for (int c = threadIdx.x; c < K; c += blockDim.x) {
                const int r = c / h;
                const int j = c - r * h;
                const float x = to_f32<kBF16>(static_cast<const uint16_t *>(chunks.p[r])[t * h + j]);
                const float y = smooth ? __fmul_rn(x, to_f32<kBF16>(smooth[c])) : x;
                const int q = quant1(y, scale);
                qrow[c] = __int2half_rn(q);
                if (orow) orow[c] = static_cast<int8_t>(q);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Fused prologue of the dynamic-quant scenario, for h % 8 == 0 and
// rank_size*h <= 32768: one launch whose CTAs take one of two roles,
// interleaved so that both run side by side on every SM --
//   * quant CTAs (one per permuted row t): one thread copies the row's
//     rank_size pieces chunk_r[t, 0:h] into shared memory with bulk async
//     copies, which lays them out as the permuted row P[t, :] (piece r at
//     columns r*h ..); both passes then read the row from shared memory, so a
//     CTA holds no row in registers and many rows are in flight per SM;
//   * widen CTAs: a contiguous slice of x2, int8 -> fp16; their number follows
//     the size of x2 (about four 16-byte vectors per thread), and CTA b is a
//     widen CTA when floor((b+1)W/G) > floor(bW/G) (W widen CTAs of G), which
//     spreads the two roles evenly over the grid.
// The quant role is instruction-bound and the widening memory-bound, which is
// why they share the launch.
//
// Rounding without a division.  With rcp = 1/scale correctly rounded,
// qa = fl(y * rcp) and the correctly rounded quotient z = fl(y / scale) are
// both within a relative 2^-23 of y / scale, and |y / scale| < 127.5, so
// |qa - z| < 2^-15.  k = fl(qa + M) - M with M = 1.5 * 2^23 is qa rounded to
// the nearest integer, ties to even (every value in [2^23, 2^24) is an
// integer and M is even), and d = qa - k is exact.  If |d| <= 0.5 - 2^-12,
// z lies strictly between k - 1/2 and k + 1/2, so rne(z) = k; otherwise (rare,
// and every exact tie) the IEEE division decides.  qa <= 127 * (1 + 3*2^-24)
// keeps k inside [-127, 127], and the low byte of fl(qa + M) is k mod 256,
// i.e. the int8 q.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
// 256 threads per CTA (one permuted row, or a widening slice): against 128,
// a2a-dyn-small 69.3 -> 65.2 us and a2a-dyn 198.3 -> 196.2 us; 512 was slower
constexpr int kPrologueThreads = 256;

// The fp32 products of two pairs of 16-bit values (x.lo * s.lo, x.hi * s.hi),
// each the product rounded once to fp32 as a multiply gives it: one
// mixed-precision fused multiply-add per element (PTX fma.f32.bf16 / .f16), the
// 16-bit inputs read straight from the packed words instead of widened first.
// Adding -0 changes no product, a zero of either sign included.  A product of
// two bf16 or fp16 values has at most 22 significant bits, so it is exact
// unless it underflows, and then both forms round it the same way.  Against
// the widening and a paired multiply: fewer instructions, and the prologue
// 47.3 -> 46.7 us on a2a-dyn, 27.1 -> 26.3 us on a2a-dyn-small (same process,
// bit-identical).
template <bool kBF16>
__device__ __forceinline__ float2 mul_exact2(uint32_t x, uint32_t s) {
    float2 y;
    if constexpr (kBF16) {
        asm("{\n\t.reg .b16 xl, xh, sl, sh;\n\t"
            "mov.b32 {xl, xh}, %2;\n\tmov.b32 {sl, sh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, xl, sl, 0f80000000;\n\t"
            "fma.rn.f32.bf16 %1, xh, sh, 0f80000000;\n\t}"
            : "=f"(y.x), "=f"(y.y)
            : "r"(x), "r"(s));
    } else {
        asm("{\n\t.reg .b16 xl, xh, sl, sh;\n\t"
            "mov.b32 {xl, xh}, %2;\n\tmov.b32 {sl, sh}, %3;\n\t"
            "fma.rn.f32.f16 %0, xl, sl, 0f80000000;\n\t"
            "fma.rn.f32.f16 %1, xh, sh, 0f80000000;\n\t}"
            : "=f"(y.x), "=f"(y.y)
            : "r"(x), "r"(s));
    }
    return y;
}

template <bool kBF16>
__device__ __forceinline__ uint4 smooth_vec(const uint16_t *smooth, int vi) {
    if (smooth) return __ldg(reinterpret_cast<const uint4 *>(smooth + vi * 8));
    return kBF16 ? make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u)    // bf16 1.0
                 : make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);   // fp16 1.0
}

template <bool kBF16>
__global__ void __launch_bounds__(kPrologueThreads) a2a_prologue_kernel(
    const __grid_constant__ ChunkPtrs chunks, int h, int64_t bs_local, int rank_size,
    const uint16_t *__restrict__ smooth, __half *__restrict__ qh, int8_t *__restrict__ q_out,
    float *__restrict__ scale_out, const int8_t *__restrict__ x2, __half *__restrict__ x2h, int64_t x2_vecs,
    int64_t widen_ctas, uint16_t *__restrict__ comm_out, int *status,
    uint64_t wait_limit_ns) {
    extern __shared__ __align__(128) uint8_t prow[];   // the permuted row (K bf16/fp16), then its mbarrier
    // launched as a programmatic dependent of the stream's previous kernel:
    // nothing in global memory is touched before that kernel has completed
    ptx::grid_dependency_wait();
    const int64_t b = blockIdx.x;
    const int64_t G = gridDim.x;
    const int64_t before = b * widen_ctas / G;  // widen CTAs among [0, b)
    if ((b + 1) * widen_ctas / G > before) {
        // ---- widen role: vectors [w * per, (w + 1) * per) of 16 int8 each
        const int64_t w = before;
        const int64_t per = (x2_vecs + widen_ctas - 1) / widen_ctas;
        const int64_t end = min(x2_vecs, (w + 1) * per);
        // two coalesced loads in flight per thread before any conversion, on many
        // short CTAs (as in widen_a2a_kernel; four per thread measured 2 µs slower on
        // a2a-dyn and a2a-dyn-small)
        for (int64_t i0 = w * per + threadIdx.x; i0 < end; i0 += 2 * blockDim.x) {
            int4 v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t i = i0 + u * blockDim.x;
                if (i < end) v[u] = __ldg(reinterpret_cast<const int4 *>(x2) + i);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t i = i0 + u * blockDim.x;
                if (i >= end) break;
                uint4 o[2];
                i8x16_to_f16x16(v[u], o);
                reinterpret_cast<uint4 *>(x2h)[2 * i] = o[0];
                reinterpret_cast<uint4 *>(x2h)[2 * i + 1] = o[1];
            }
        }
        ptx::allow_dependent_launch();
        return;
    }
    // ---- quant role: permuted row t
    const int64_t t = b - before;
    if (t >= bs_local) {
        ptx::allow_dependent_launch();
        return;
    }
    __shared__ float red[32];
    const int K = rank_size * h;
    const int nvec = K / 8;
    const uint32_t row_s = ptx::smem_u32(prow);
    const uint32_t bar = row_s + static_cast<uint32_t>(K) * 2u;   // K * 2 is a multiple of 16
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(K) * 2u);
        for (int r = 0; r < rank_size; ++r)
            ptx::bulk_load_1d(row_s + static_cast<uint32_t>(r * h) * 2u,
                              static_cast<const uint16_t *>(chunks.p[r]) + t * h, static_cast<uint32_t>(h) * 2u, bar);
    }
    __syncthreads();   // the barrier is initialised before anyone polls it
    // A thread whose bounded wait gives up raises the status word and still
    // takes part in the row (its outputs are void then): the threads' waits can
    // end on either side of the limit, and one that left early would strand the
    // others at the row's block barriers.
    if (!ptx::mbar_wait(bar, 0, wait_limit_ns) && status) atomicExch(status, -7);
    const uint4 *rowv = reinterpret_cast<const uint4 *>(prow);
    // commOut: the received pieces in their own layout (rank_size, bs_local, h)
    if (comm_out) {
        for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
            const int c = vi * 8;
            const int r = c / h;
            *reinterpret_cast<uint4 *>(comm_out + (r * bs_local + t) * h + (c - r * h)) = rowv[vi];
        }
    }
    // y = x * s (fp32, exact for 16-bit inputs); row absmax
    float amax = 0.0f;
    for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
        const uint4 xv = rowv[vi];
        const uint4 sv = smooth_vec<kBF16>(smooth, vi);
        const uint32_t *xw = reinterpret_cast<const uint32_t *>(&xv);
        const uint32_t *sw = reinterpret_cast<const uint32_t *>(&sv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 y = mul_exact2<kBF16>(xw[e], sw[e]);
            amax = fmaxf(amax, fmaxf(fabsf(y.x), fabsf(y.y)));
        }
    }
    amax = block_max(amax, red);
    const float scale = __fdiv_rn(amax, 127.0f);
    const float rcp = scale == 0.0f ? 0.0f : __frcp_rn(scale);
    const bool row_fast = rcp <= 3.0e38f;  // 1/scale finite (always, unless amax is subnormal)
    if (threadIdx.x == 0) scale_out[t] = scale;
    const float2 rcp2 = make_float2(rcp, rcp);
    const float2 magic2 = make_float2(kRoundMagic, kRoundMagic);
    const float2 nmagic2 = make_float2(-kRoundMagic, -kRoundMagic);
    for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
        const uint4 xv = rowv[vi];
        const uint4 sv = smooth_vec<kBF16>(smooth, vi);
        const uint32_t *xw = reinterpret_cast<const uint32_t *>(&xv);
        const uint32_t *sw = reinterpret_cast<const uint32_t *>(&sv);
        uint4 hv;
        __half2 *hh = reinterpret_cast<__half2 *>(&hv);
        uint32_t qb[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 y = mul_exact2<kBF16>(xw[e], sw[e]);
            const float2 qa = __fmul2_rn(y, rcp2);
            const float2 tm = __fadd2_rn(qa, magic2);   // M + rne(qa)
            const float2 k = __fadd2_rn(tm, nmagic2);   // rne(qa), exact
            const float2 d = __fadd2_rn(qa, make_float2(-k.x, -k.y));
            float2 kq = k;
            uint32_t b0 = __float_as_uint(tm.x), b1 = __float_as_uint(tm.y);
            if (!row_fast || fmaxf(fabsf(d.x), fabsf(d.y)) > 0.499755859375f) {
                const int q0 = quant1(y.x, scale), q1 = quant1(y.y, scale);
                kq = make_float2(static_cast<float>(q0), static_cast<float>(q1));
                b0 = static_cast<uint32_t>(q0);
                b1 = static_cast<uint32_t>(q1);
            }
            hh[e] = __float22half2_rn(kq);
            qb[2 * e] = b0;
            qb[2 * e + 1] = b1;
        }
        *reinterpret_cast<uint4 *>(qh + t * K + vi * 8) = hv;
        if (q_out) {
            uint2 iv;
            iv.x = __byte_perm(__byte_perm(qb[0], qb[1], 0x0040), __byte_perm(qb[2], qb[3], 0x0040), 0x5410);
            iv.y = __byte_perm(__byte_perm(qb[4], qb[5], 0x0040), __byte_perm(qb[6], qb[7], 0x0040), 0x5410);
            *reinterpret_cast<uint2 *>(q_out + t * K + vi * 8) = iv;
        }
    }
    // The GEMM that follows is launched once every CTA of this grid has got here
    // (it still waits for the whole grid to finish before reading): triggering
    // at the end, not the start, keeps its CTAs, which need a whole SM, from
    // taking SMs that the remaining CTAs of this grid still need.
    ptx::allow_dependent_launch();
}

// int8 -> fp16, exact.  Each warp moves 64 consecutive 16-element vectors per
// step (two coalesced 16-byte loads per lane in flight), on a large grid (see
// widen_a2a_kernel); the count % 16 elements past the last vector one by one.
__global__ void __launch_bounds__(256) widen_i8_kernel(const int8_t *__restrict__ src, __half *__restrict__ dst,
                                                       int64_t count) {
    const int64_t nvec = count / 16;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp0 * 64; base < nvec; base += nwarps * 64) {
        int4 v[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t i = base + 32 * j + lane;
            if (i < nvec) v[j] = __ldg(reinterpret_cast<const int4 *>(src) + i);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t i = base + 32 * j + lane;
            if (i >= nvec) continue;
            uint4 o[2];
            i8x16_to_f16x16(v[j], o);
            reinterpret_cast<uint4 *>(dst)[2 * i] = o[0];
            reinterpret_cast<uint4 *>(dst)[2 * i + 1] = o[1];
        }
    }
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = nvec * 16 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += stride)
        dst[i] = __int2half_rn(src[i]);
    // the GEMM that follows launches once every CTA got here (see a2a_prologue_kernel)
    ptx::allow_dependent_launch();
}

// The full-quant path's two widenings in one launch: each rank's int8 chunk
// -> fp16 in its own layout at dst_a + r * bs_local * h (the GEMM then reads
// the permuted matrix through one tensor map per chunk instead of a permuted
// copy), and x2 (K, n) int8 -> fp16 (dst_b); q_out (optional) gets the permuted
// int8 matrix.  The two are one vector
// space of 16-element vectors: [0, total_a) the chunks, [total_a, total_a +
// total_b) x2.  Each warp moves 64 consecutive vectors per step, lane l taking
// vectors l and l + 32, so each 16-byte load is a coalesced 512 bytes and both
// are in flight before the first conversion, and the grid is large (up to 128
// CTAs per SM, most of them one step long).  On a2a-full that measured 376 µs
// (90% of the copy rate) against 537 µs for four vectors per lane on a grid of
// 8 CTAs per SM and 464–471 µs for other mixes.  h % 16 == 0 and n % 16 == 0.
__global__ void __launch_bounds__(256) widen_a2a_kernel(const __grid_constant__ ChunkPtrs chunks, int h,
                                                        int64_t bs_local, int rank_size, __half *__restrict__ dst_a,
                                                        const int8_t *__restrict__ x2, __half *__restrict__ dst_b,
                                                        int64_t total_b, int8_t *__restrict__ q_out,
                                                        int8_t *__restrict__ comm_out) {
    const int64_t per_chunk = bs_local * h / 16;
    const int64_t total_a = per_chunk * rank_size;
    const int64_t total = total_a + total_b;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int vpr = h / 16;
    for (int64_t base = warp0 * 64; base < total; base += nwarps * 64) {
        int4 v[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t i = base + 32 * j + lane;
            if (i < total_a) {
                const int r = static_cast<int>(i / per_chunk);
                v[j] = __ldg(reinterpret_cast<const int4 *>(chunks.p[r]) + (i - r * per_chunk));
            } else if (i < total) {
                v[j] = __ldg(reinterpret_cast<const int4 *>(x2) + (i - total_a));
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t i = base + 32 * j + lane;
            if (i >= total) continue;
            uint4 o[2];
            i8x16_to_f16x16(v[j], o);
            if (i < total_a) {
                uint4 *d = reinterpret_cast<uint4 *>(dst_a) + 2 * i;
                d[0] = o[0];
                d[1] = o[1];
                // commOut (rank_size, bs_local, h) is the chunks back to back: vector i
                if (comm_out) reinterpret_cast<int4 *>(comm_out)[i] = v[j];
                if (q_out) {
                    const int r = static_cast<int>(i / per_chunk);
                    const int64_t li = i - r * per_chunk;
                    const int64_t t = li / vpr;
                    const int c = static_cast<int>(li - t * vpr) * 16;
                    *reinterpret_cast<int4 *>(q_out + t * (static_cast<int64_t>(rank_size) * h) + r * h + c) = v[j];
                }
            } else {
                uint4 *d = reinterpret_cast<uint4 *>(dst_b) + 2 * (i - total_a);
                d[0] = o[0];
                d[1] = o[1];
            }
        }
    }
    // the GEMM that follows launches once every CTA got here (see a2a_prologue_kernel)
    ptx::allow_dependent_launch();
}

// Permuted int8 chunks -> fp16 GEMM operand (and optionally the int8
// permuted matrix): dst[t, r*h + j] = chunk_r[t, j].
__global__ void __launch_bounds__(256) permute_widen_i8_kernel(const __grid_constant__ ChunkPtrs chunks, int h, int64_t bs_local,
                                                               int rank_size, __half *__restrict__ dst,
                                                               int8_t *__restrict__ q_out,
                                                               int8_t *__restrict__ comm_out) {
    ptx::allow_dependent_launch();
    const int K = rank_size * h;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (h % 16 == 0) {
        const int vpr = K / 16;
        const int64_t total = bs_local * vpr;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
            const int64_t t = i / vpr;
            const int c = static_cast<int>(i - t * vpr) * 16;
            const int r = c / h;
            const int j = c - r * h;
            const int4 v = __ldg(reinterpret_cast<const int4 *>(static_cast<const int8_t *>(chunks.p[r]) + t * h + j));
            uint4 o[2];
            i8x16_to_f16x16(v, o);
            uint4 *d = reinterpret_cast<uint4 *>(dst + t * K + c);
            d[0] = o[0];
            d[1] = o[1];
            if (q_out) *reinterpret_cast<int4 *>(q_out + t * K + c) = v;
            if (comm_out) *reinterpret_cast<int4 *>(comm_out + (r * bs_local + t) * h + j) = v;
        }
    } else {
        const int64_t total = bs_local * K;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
            const int64_t t = i / K;
            const int c = static_cast<int>(i - t * K);
            const int r = c / h;
            const int j = c - r * h;
            const int8_t v = static_cast<const int8_t *>(chunks.p[r])[t * h + j];
            dst[i] = __int2half_rn(v);
            if (q_out) q_out[i] = v;
            if (comm_out) comm_out[(r * bs_local + t) * h + j] = v;
        }
    }
}

int grid_for(int64_t work_items, int threads, int num_sms) {
    int64_t g = (work_items + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_quant_pertoken(const ChunkPtrs &chunks, int rank_size, int64_t bs_local, int h, bool bf16,
                                  const void *smooth, __half *qh, int8_t *q_out, float *scale_out, void *comm_out,
                                  int num_sms, cudaStream_t stream) {
    uint16_t *co = static_cast<uint16_t *>(comm_out);
    const uint16_t *sm = static_cast<const uint16_t *>(smooth);
    const int64_t rows_cap = static_cast<int64_t>(num_sms) * 64;
    const int grid = static_cast<int>(bs_local < rows_cap ? bs_local : rows_cap);
    if (bf16)
        quant_pertoken_kernel<true><<<grid, 256, 0, stream>>>(chunks, h, bs_local, rank_size, sm, qh, q_out,
                                                              scale_out, co);
    else
        quant_pertoken_kernel<false><<<grid, 256, 0, stream>>>(chunks, h, bs_local, rank_size, sm, qh, q_out,
                                                               scale_out, co);
    return cudaGetLastError();
}

bool a2a_prologue_fits(int rank_size, int64_t bs_local, int h) {
    return h % 8 == 0 && static_cast<int64_t>(rank_size) * h <= 512 * 64 && bs_local <= (1ll << 30);
}

cudaError_t launch_a2a_prologue(const ChunkPtrs &chunks, int rank_size, int64_t bs_local, int h, bool bf16,
                                const void *smooth, __half *qh, int8_t *q_out, float *scale_out, const int8_t *x2,
                                __half *x2h, int64_t x2_count, void *comm_out,
                                int *status, uint64_t wait_limit_ns, cudaStream_t stream) {
    uint16_t *co = static_cast<uint16_t *>(comm_out);
    const int K = rank_size * h;
    constexpr int threads = kPrologueThreads;
    // the permuted row and its mbarrier
    const size_t smem = static_cast<size_t>(K) * 2 + 16;
    // one quant CTA per row; widen CTAs for ~4 vectors per thread
    const int64_t x2_vecs = x2_count / 16;
    int64_t widen_ctas = (x2_vecs + 2ll * threads - 1) / (2ll * threads);
    if (widen_ctas < 1) widen_ctas = 1;
    if (widen_ctas > (1ll << 30)) widen_ctas = 1ll << 30;
    const int64_t grid = bs_local + widen_ctas;
    const uint16_t *sm = static_cast<const uint16_t *>(smooth);
    auto kern = bf16 ? a2a_prologue_kernel<true> : a2a_prologue_kernel<false>;
    // rows above 48 KiB need the opt-in (raised once per host thread, context and type)
    thread_local unsigned long long opted_ctx[2] = {0, 0};
    if (smem > 48 * 1024) {
        const unsigned long long ctx = current_context_id();
        if (ctx == 0 || ctx != opted_ctx[bf16 ? 1 : 0]) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024 + 16);
            if (e != cudaSuccess) return e;
            opted_ctx[bf16 ? 1 : 0] = ctx;
        }
    }
    // its CTAs may be scheduled before the previous kernel ends (they wait for it)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, chunks, h, bs_local, rank_size, sm, qh, q_out, scale_out, x2, x2h,
                                       x2_vecs, widen_ctas, co, status, wait_limit_ns);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_widen_i8(const int8_t *src, __half *dst, int64_t count, int num_sms, cudaStream_t stream) {
    // one step of 8 warps x 64 vectors per CTA, up to 128 CTAs per SM
    int64_t grid = (count / 16 + 8 * 64 - 1) / (8 * 64);
    const int64_t cap = static_cast<int64_t>(num_sms) * 128;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    widen_i8_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(src, dst, count);
    return cudaGetLastError();
}

cudaError_t launch_widen_a2a(const ChunkPtrs &chunks, int rank_size, int64_t bs_local, int h, __half *dst_a,
                             const int8_t *x2, __half *dst_b, int64_t x2_count, int8_t *q_out, int8_t *comm_out,
                             int num_sms, cudaStream_t stream) {
    const int64_t total = bs_local * static_cast<int64_t>(rank_size) * h / 16 + x2_count / 16;
    // one step of 8 warps x 64 vectors per CTA, up to 128 CTAs per SM
    int64_t grid = (total + 8 * 64 - 1) / (8 * 64);
    const int64_t cap = static_cast<int64_t>(num_sms) * 128;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    widen_a2a_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(chunks, h, bs_local, rank_size, dst_a, x2, dst_b,
                                                                      x2_count / 16, q_out, comm_out);
    return cudaGetLastError();
}

cudaError_t launch_permute_widen_i8(const ChunkPtrs &chunks, int rank_size, int64_t bs_local, int h, __half *dst,
                                    int8_t *q_out, int8_t *comm_out, int num_sms, cudaStream_t stream) {
    const int64_t items = bs_local * static_cast<int64_t>(rank_size) * h / ((h % 16 == 0) ? 16 : 1);
    permute_widen_i8_kernel<<<grid_for(items, 256, num_sms), 256, 0, stream>>>(chunks, h, bs_local, rank_size, dst,
                                                                              q_out, comm_out);
    return cudaGetLastError();
}

}  // namespace mc2
