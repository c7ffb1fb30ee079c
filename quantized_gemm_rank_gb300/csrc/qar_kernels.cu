// qar_kernels.cu -- QuantAllReduce ("QuantAllReduce", ops-transformer
// mc2/quant_all_reduce, 功能说明: output = Reduce(AllGather(scales) *
// AllGather(x)) with reduceOp "sum"; 参数说明/约束说明: x int8, fp8 e4m3fn or
// fp8 e5m2; scales fp32 per token per group of 128 (pertoken-pergroup) or
// e8m0 per group of 32 stored (bs, H/64, 2) (mx); H in [1024, 8192], a
// multiple of 128).
//
// Every rank's (x_r, scales_r) is a separate device buffer on this GPU, so the
// all-gather is addressing and the reduce is a sum in registers:
//   out[t, j] = sum_r dec(x_r[t, j]) * dec(scales_r[t, j / G])
// The products are added in rank order by fp32 fused multiply-adds and the sum
// is rounded once (nearest-even) to the output type.
//
// HBM-bound: each rank's codes are read once (16-byte loads with a 256-byte L2
// fetch, one or two per rank in flight per thread), the output written once.  Because G divides H,
// the scale of flat element e is scales_r[e / G] whatever the row, so the
// kernel runs over the flat (bs * H) range with no row arithmetic.
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "internal.h"

namespace mc2 {

namespace {

constexpr int kVec = 16;          // one-byte codes per vector (one 16-byte load per rank)
constexpr int kThreads = 256;

// int8 code -> float without a conversion instruction: flipping the sign bit
// gives x + 128 in [0, 255]; placed in the low mantissa byte of 2^23 that is
// the float 2^23 + x + 128, and subtracting 2^23 + 128 leaves x exactly.
__device__ __forceinline__ void decode_i8(const uint4 &v, float (&f)[kVec]) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t b = w[e] ^ 0x80808080u;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[4 * e + i] = __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7540u + i)) - 8388736.0f;
    }
}

// fp8 pairs -> f16 pairs (exact: every e4m3fn and e5m2 value, subnormals and
// e5m2 infinities included, is a half) -> float.
template <bool kE5M2>
__device__ __forceinline__ void decode_f8(const uint4 &v, float (&f)[kVec]) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>(w[e] >> (16 * i));
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, kE5M2 ? __NV_E5M2 : __NV_E4M3);
            const float2 ff = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
            f[4 * e + 2 * i] = ff.x;
            f[4 * e + 2 * i + 1] = ff.y;
        }
    }
}

// e8m0 scale code c -> 2^(c - 127): the code is the float's exponent field;
// c == 0 is 2^-127, a subnormal; c == 0xFF is NaN.
__device__ __forceinline__ float decode_e8m0(uint32_t c) {
    if (c == 0u) return __uint_as_float(0x00400000u);
    if (c == 0xFFu) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(c << 23);
}

struct QarPtrs {
    const uint8_t *x[8];
    const void *s[8];
};

// One vector: 16 elements of every rank, summed and stored.
template <int kX, int kS, int kOut, int kR>
__device__ __forceinline__ void reduce_store(const uint4 (&xv)[kR], const float (&sc)[kR], void *__restrict__ out,
                                             int64_t v) {
    float acc[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;   // the sum starts at +0, as the reduction's definition
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        float f[kVec];
        if constexpr (kX == 0)
            decode_i8(xv[r], f);
        else
            decode_f8<kX == 2>(xv[r], f);
#pragma unroll
        for (int i = 0; i < kVec; ++i) acc[i] = __fmaf_rn(f[i], sc[r], acc[i]);
    }
    if constexpr (kOut == 0) {
        float4 *o = reinterpret_cast<float4 *>(out) + v * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            __stcs(o + q, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
    } else {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if constexpr (kOut == 1) {
                const __half2 h2 = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t *>(&h2);
            } else {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t *>(&b2);
            }
        }
        uint4 *o = reinterpret_cast<uint4 *>(out) + v * 2;
        __stcs(o, make_uint4(w[0], w[1], w[2], w[3]));
        __stcs(o + 1, make_uint4(w[4], w[5], w[6], w[7]));
    }
}

// A 16-byte load of codes that are read once: through the read-only path, not
// allocated in L1, with L2 asked to fetch the whole 256-byte block around it
// from DRAM (the L2::256B prefetch-size qualifier), so a warp's 512 contiguous
// bytes arrive as two whole blocks.  With one such stream per rank in flight
// this measured 62.1 -> 58.5 us on qar-8x4096x8192 against evict-first loads
// (same process, bit-identical); the widening kernels, with one or two streams,
// gained nothing from it.
__device__ __forceinline__ uint4 ld_code_vec(const uint4 *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

template <int kS, int kR>
__device__ __forceinline__ void load_vec(const QarPtrs &p, int64_t v, uint4 (&xv)[kR], float (&sc)[kR]) {
#pragma unroll
    for (int r = 0; r < kR; ++r) xv[r] = ld_code_vec(reinterpret_cast<const uint4 *>(p.x[r]) + v);
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        if constexpr (kS == 0)
            sc[r] = __ldg(static_cast<const float *>(p.s[r]) + (v >> 3));                  // G = 128 = 8 vectors
        else
            sc[r] = decode_e8m0(__ldg(static_cast<const uint8_t *>(p.s[r]) + (v >> 1)));  // G = 32
    }
}

// kX: 0 int8, 1 e4m3fn, 2 e5m2.  kS: 0 fp32 per 128, 1 e8m0 per 32.
// kOut: 0 fp32, 1 fp16, 2 bf16.  kR: ranks.  With int8 codes each thread
// takes two vectors per step (v and v + stride, the loads of both in flight
// before either is reduced); the fp8 decode needs more registers, and there
// one vector per step keeps more threads resident.  The launch bound asks for 4
// CTAs per SM (64 registers): at the 80 registers the compiler chose otherwise,
// 3 fit, and the loads in flight of the 4th are worth more than the registers
// (qar-8x4096x8192: 68.2 -> 62.1 us; 6 CTAs at 40 registers spill and run slower).
template <int kX, int kS, int kOut, int kR>
__global__ void __launch_bounds__(kThreads, 4) quant_all_reduce_kernel(QarPtrs p, int64_t nvec, void *__restrict__ out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t v = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if constexpr (kX == 0) {
        for (; v + stride < nvec; v += 2 * stride) {
            uint4 xa[kR], xb[kR];
            float sa[kR], sb[kR];
            load_vec<kS, kR>(p, v, xa, sa);
            load_vec<kS, kR>(p, v + stride, xb, sb);
            reduce_store<kX, kS, kOut, kR>(xa, sa, out, v);
            reduce_store<kX, kS, kOut, kR>(xb, sb, out, v + stride);
        }
    }
    for (; v < nvec; v += stride) {
        uint4 xa[kR];
        float sa[kR];
        load_vec<kS, kR>(p, v, xa, sa);
        reduce_store<kX, kS, kOut, kR>(xa, sa, out, v);
    }
}

template <int kX, int kS, int kOut, int kR>
cudaError_t launch_one(const QarPtrs &p, int64_t nvec, void *out, int num_sms, cudaStream_t stream) {
    // Persistent grid: as many CTAs as fit on the device at once (the
    // occupancy of this instantiation, looked up once per process).
    static std::atomic<int> per_sm_cache{0};
    int per_sm = per_sm_cache.load(std::memory_order_relaxed);
    if (per_sm == 0) {
        int b = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &b, quant_all_reduce_kernel<kX, kS, kOut, kR>, kThreads, 0);
        if (e != cudaSuccess) return e;
        per_sm = b > 0 ? b : 1;
        per_sm_cache.store(per_sm, std::memory_order_relaxed);
    }
    const int64_t need = (nvec + kThreads - 1) / kThreads;
    const int64_t full = static_cast<int64_t>(num_sms) * per_sm;
    const unsigned grid = static_cast<unsigned>(need < full ? need : full);
    quant_all_reduce_kernel<kX, kS, kOut, kR><<<grid, kThreads, 0, stream>>>(p, nvec, out);
    return cudaGetLastError();
}

template <int kX, int kS, int kOut>
cudaError_t dispatch_r(int ranks, const QarPtrs &p, int64_t nvec, void *out, int num_sms, cudaStream_t s) {
    switch (ranks) {
        case 2: return launch_one<kX, kS, kOut, 2>(p, nvec, out, num_sms, s);
        case 4: return launch_one<kX, kS, kOut, 4>(p, nvec, out, num_sms, s);
        case 8: return launch_one<kX, kS, kOut, 8>(p, nvec, out, num_sms, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int kX, int kS>
cudaError_t dispatch_out(int out_kind, int ranks, const QarPtrs &p, int64_t nvec, void *out, int num_sms,
                         cudaStream_t s) {
    switch (out_kind) {
        case 0: return dispatch_r<kX, kS, 0>(ranks, p, nvec, out, num_sms, s);
        case 1: return dispatch_r<kX, kS, 1>(ranks, p, nvec, out, num_sms, s);
        case 2: return dispatch_r<kX, kS, 2>(ranks, p, nvec, out, num_sms, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_quant_all_reduce(const void *const *x_chunks, const void *const *scale_chunks, int ranks,
                                    int64_t elems, int x_kind, int scale_kind, int out_kind, void *out, int num_sms,
                                    cudaStream_t stream) {
    if (ranks < 1 || ranks > 8 || elems % kVec != 0) return cudaErrorInvalidValue;
    QarPtrs p{};
    for (int r = 0; r < ranks; ++r) {
        p.x[r] = static_cast<const uint8_t *>(x_chunks[r]);
        p.s[r] = scale_chunks[r];
    }
    const int64_t nvec = elems / kVec;
    if (scale_kind == 0) {
        switch (x_kind) {
            case 0: return dispatch_out<0, 0>(out_kind, ranks, p, nvec, out, num_sms, stream);
            case 1: return dispatch_out<1, 0>(out_kind, ranks, p, nvec, out, num_sms, stream);
            case 2: return dispatch_out<2, 0>(out_kind, ranks, p, nvec, out, num_sms, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (x_kind) {
        case 1: return dispatch_out<1, 1>(out_kind, ranks, p, nvec, out, num_sms, stream);
        case 2: return dispatch_out<2, 1>(out_kind, ranks, p, nvec, out, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mc2
