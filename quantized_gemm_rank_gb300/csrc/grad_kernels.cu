// grad_kernels.cu -- the bias gradient of the fused linear layers
// ("hyper_parallel .../mc2.py", AllGatherMatmulFunction.backward:
// grad_bias = grad_out.sum(dim=0)): the column sums of dY (m, n), accumulated
// in fp32 and rounded once to dY's 16-bit type.  HBM-bound: every element of
// dY is read once, with 16-byte loads, eight in flight per thread.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mc2 {

namespace {

constexpr int kStripCols = 32;   // columns per CTA: 4 vectors of 8
constexpr int kRowLanes = 64;    // threads down the rows of one vector column
constexpr int kUnroll = 8;

template <bool kBF16>
__device__ __forceinline__ void add8(float (&acc)[8], const uint4 &v) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float lo, hi;
        if constexpr (kBF16) {
            lo = __uint_as_float(w[e] << 16);
            hi = __uint_as_float(w[e] & 0xFFFF0000u);
        } else {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
            lo = f.x;
            hi = f.y;
        }
        acc[2 * e] += lo;
        acc[2 * e + 1] += hi;
    }
}

// One CTA per strip of 32 columns (n % 8 == 0, so a vector is wholly in or
// out).  Thread (lane_r, vc) sums rows lane_r, lane_r + 64, ... of vector vc;
// the 64 partial sums of a column are then added in lane order.
template <bool kBF16>
__global__ void __launch_bounds__(256) colsum16_kernel(const uint16_t *__restrict__ dy, int64_t m, int n,
                                                       uint16_t *__restrict__ db) {
    ptx::allow_dependent_launch();
    __shared__ float red[kRowLanes][kStripCols + 1];
    const int vc = threadIdx.x & 3;
    const int lane_r = threadIdx.x >> 2;
    const int col0 = blockIdx.x * kStripCols + vc * 8;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    if (col0 < n) {
        const uint16_t *base = dy + col0;
        int64_t t = lane_r;
        for (; t + (kUnroll - 1) * kRowLanes < m; t += kUnroll * kRowLanes) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                v[u] = __ldg(reinterpret_cast<const uint4 *>(base + (t + u * kRowLanes) * n));
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) add8<kBF16>(acc, v[u]);
        }
        for (; t < m; t += kRowLanes) add8<kBF16>(acc, __ldg(reinterpret_cast<const uint4 *>(base + t * n)));
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) red[lane_r][vc * 8 + e] = acc[e];
    __syncthreads();
    if (threadIdx.x < kStripCols) {
        const int col = blockIdx.x * kStripCols + threadIdx.x;
        float s = 0.0f;
        for (int l = 0; l < kRowLanes; ++l) s += red[l][threadIdx.x];
        if (col < n) {
            if constexpr (kBF16)
                db[col] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
            else
                db[col] = __half_as_ushort(__float2half_rn(s));
        }
    }
}

}  // namespace

cudaError_t launch_colsum16(const void *dy, int64_t m, int n, bool bf16, void *db, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>((n + kStripCols - 1) / kStripCols);
    const uint16_t *src = static_cast<const uint16_t *>(dy);
    uint16_t *dst = static_cast<uint16_t *>(db);
    if (bf16)
        colsum16_kernel<true><<<grid, 256, 0, stream>>>(src, m, n, dst);
    else
        colsum16_kernel<false><<<grid, 256, 0, stream>>>(src, m, n, dst);
    return cudaGetLastError();
}

}  // namespace mc2
