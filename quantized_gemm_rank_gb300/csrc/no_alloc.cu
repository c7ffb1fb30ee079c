// no_alloc.cu -- AlltoAllQuantMatmul for callers that cannot allocate device
// memory.
//
// The regular entry point asks the caller for a workspace.  Some callers have
// no way to provide one:
//   - a C or Fortran host program that links only this library and owns no
//     device allocator;
//   - a plugin inside a framework that owns all device memory and forbids its
//     plugins to call cudaMalloc.  cudaMalloc can synchronise the whole device,
//     and it fragments the framework's own pool.
// This entry point gives those callers the same computation with the scratch
// held in a fixed, file-scope device array instead.
//
// Costs and rules of that array:
//   - It is kMaxScratchBytes (32 MiB) on every GPU that loads this library, and
//     stays allocated until the process exits.  Under CUDA's lazy module
//     loading (the default) the library's device code, this array with it, is
//     loaded on a device the first time the library is used there, so the
//     first call on a device maps the 32 MiB; a caller that must not see
//     device memory grow mid-run makes one warm-up call at start-up.
//   - Every call shares it, so calls whose work overlaps on the GPU (different
//     streams, or different host threads) race on it.  Serialise them.
//   - It keeps whatever the last call left there.  Nothing in it has to start at
//     zero: every byte the kernels read is written earlier in the same call
//     (the stream-K flags carry a per-launch epoch, so stale ones count as none).
#include <cuda_runtime.h>

#include <cstdio>

#include "internal.h"
#include "mc2_gb300.h"

namespace {

constexpr size_t kMaxScratchBytes = MC2_NO_ALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_no_alloc_scratch[kMaxScratchBytes];

// Device address of g_no_alloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the real address is looked
// up with the device current.  It is looked up on every call: the lookup
// neither allocates nor synchronises, and an address kept from before a
// device reset would point into a context that no longer exists.
int scratch_for_current_device(void **ptr) {
    char msg[160];
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the scratch failed: %s", cudaGetErrorString(e));
        return mc2::record_error(MC2_ERR_CUDA, msg);
    }
    *ptr = p;
    return MC2_OK;
}

}  // namespace

extern "C" int mc2_alltoall_quant_mm_no_alloc(const void *const *chunks, int rank_size, int64_t bs_local,
                                              int64_t h, int x1_dtype, const void *x1_scale, const int8_t *x2,
                                              const float *x2_scale, const void *bias, int bias_dtype,
                                              int x1_quant_mode, int x2_quant_mode, int64_t n, void *out,
                                              void *alltoall_out, int8_t *q_out, float *x1_scale_out,
                                              int32_t *acc_out, void *stream) {
    // Sizes are checked (and the scratch need computed) on the host first, so a
    // request that does not fit is refused before any device work.
    size_t need = 0;
    int st = mc2_alltoall_quant_mm_workspace(rank_size, bs_local, h, n, x1_quant_mode, x1_dtype, &need);
    if (st != MC2_OK) return st;
    if (need > kMaxScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "these sizes need %zu bytes of scratch; the built-in scratch holds %zu (MC2_NO_ALLOC_SCRATCH_BYTES)",
                 need, kMaxScratchBytes);
        return mc2::record_error(MC2_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    st = scratch_for_current_device(&scratch);
    if (st != MC2_OK) return st;
    return mc2_alltoall_quant_mm(chunks, rank_size, bs_local, h, x1_dtype, x1_scale, x2, x2_scale, bias, bias_dtype,
                                 x1_quant_mode, x2_quant_mode, n, out, alltoall_out, q_out, x1_scale_out, acc_out, scratch,
                                 kMaxScratchBytes, stream);
}
