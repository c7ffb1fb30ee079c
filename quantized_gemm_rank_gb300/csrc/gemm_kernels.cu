// gemm_kernels.cu -- instantiations and launch of the fused MC2 GEMM.
#include "gemm_tcgen05.cuh"
#include "internal.h"

namespace mc2 {

__device__ int g_gemm_status = 0;

namespace {

template <bool kBF16, bool kIntPath>
cudaError_t launch_one(const GemmParams &p_in, int num_sms, cudaStream_t stream) {
    auto kern = mc2_gemm_kernel<kBF16, kIntPath>;
    GemmParams p = p_in;
    cudaError_t es = cudaGetSymbolAddress(reinterpret_cast<void **>(&p.status), g_gemm_status);
    if (es != cudaSuccess) return es;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int num_tiles = ((p.m + kBM - 1) / kBM) * ((p.n + kBN - 1) / kBN);
    const int grid = num_tiles < num_sms ? num_tiles : num_sms;
    kern<<<grid, kNumThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(GemmKind kind, const GemmParams &p, int num_sms, cudaStream_t stream) {
    switch (kind) {
        case GEMM_F16: return launch_one<false, false>(p, num_sms, stream);
        case GEMM_BF16: return launch_one<true, false>(p, num_sms, stream);
        case GEMM_INT_AS_F16: return launch_one<false, true>(p, num_sms, stream);
    }
    return cudaErrorInvalidValue;
}

int gemm_smem_bytes() { return static_cast<int>(kSmemBytes); }

int read_and_clear_gemm_status(int *status) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_gemm_status, sizeof(int));
    if (e != cudaSuccess) return -1;
    e = cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(int));
    return e == cudaSuccess ? 0 : -1;
}

}  // namespace mc2
