// calib_kernels.cu -- calibration of the legacy warp-level tensor-core path
// (mma.sync) on this GPU: int8 x int8 -> int32 (m16n8k32) and fp16 x fp16 ->
// fp32 (m16n8k16).  The rates give context to the integer path's design: it
// runs int8 operands as exact fp16 through tcgen05 rather than through an int8
// tensor-core instruction.  Each warp runs kChains independent accumulator
// chains over fixed register operands (the values do not matter for the rate);
// one store per thread keeps the work live.
//
// This is a measurement probe for the benchmark, not part of the operations:
// it is built into its own library (libmc2_calib.so), which only bench.py
// loads.  Its one entry point:
//
//   int mc2_calib_mma_sync(int kind, int64_t iters, int blocks, int32_t *sink,
//                          void *stream, double *ops);
//
// launches `blocks` CTAs of 256 threads on `stream` (a cudaStream_t), each warp
// running `iters` rounds of 8 independent mma.sync on register operands:
// kind 0 = int8 x int8 -> int32 (m16n8k32), kind 1 = fp16 x fp16 -> fp32
// (m16n8k16).  `sink` (device, blocks * 256 int32) receives one word per
// thread; *ops receives the operations (2 per multiply-add) of the launch.
// Returns 0, -1 for a NULL sink or ops, -2 for a bad kind, iters or blocks,
// -6 if the launch fails.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kCalibThreads = 256;
constexpr int kChains = 8;

template <bool kS8>
__global__ void __launch_bounds__(kCalibThreads) mma_sync_rate_kernel(int64_t iters, int32_t *sink) {
    uint32_t a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = 0x3c003c00u ^ (threadIdx.x + 17u * i);
#pragma unroll
    for (int i = 0; i < 2; ++i) b[i] = 0x3c003c00u ^ (threadIdx.x + 29u * i);
    uint32_t acc = 0;
    if constexpr (kS8) {
        int32_t d[kChains][4] = {};
        for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
            for (int c = 0; c < kChains; ++c)
                asm volatile(
                    "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                    "{%0,%1,%2,%3};"
                    : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
                    : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
        }
#pragma unroll
        for (int c = 0; c < kChains; ++c) acc += static_cast<uint32_t>(d[c][0] ^ d[c][1] ^ d[c][2] ^ d[c][3]);
    } else {
        float d[kChains][4] = {};
        for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
            for (int c = 0; c < kChains; ++c)
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                    "{%0,%1,%2,%3};"
                    : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
                    : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
        }
#pragma unroll
        for (int c = 0; c < kChains; ++c)
            acc += __float_as_uint(d[c][0]) ^ __float_as_uint(d[c][1]) ^ __float_as_uint(d[c][2]) ^
                   __float_as_uint(d[c][3]);
    }
    sink[static_cast<int64_t>(blockIdx.x) * kCalibThreads + threadIdx.x] = static_cast<int32_t>(acc);
}

}  // namespace

extern "C" {

int mc2_calib_mma_sync(int kind, int64_t iters, int blocks, int32_t *sink, void *stream, double *ops) {
    if (!sink || !ops) return -1;
    if ((kind != 0 && kind != 1) || iters < 1 || blocks < 1) return -2;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kind == 0)
        mma_sync_rate_kernel<true><<<blocks, kCalibThreads, 0, s>>>(iters, sink);
    else
        mma_sync_rate_kernel<false><<<blocks, kCalibThreads, 0, s>>>(iters, sink);
    if (cudaGetLastError() != cudaSuccess) return -6;
    const double per_mma = kind == 0 ? 2.0 * 16 * 8 * 32 : 2.0 * 16 * 8 * 16;
    *ops = per_mma * kChains * static_cast<double>(iters) * (kCalibThreads / 32) * blocks;
    return 0;
}

}  // extern "C"
