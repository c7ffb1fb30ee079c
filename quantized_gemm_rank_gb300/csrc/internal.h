// internal.h -- declarations shared by the library's translation units
// (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mc2 {

struct ChunkPtrs {
    const void *p[8];
};

struct GemmParams;

// GEMM launch: kind selects the instantiation.
// GEMM_RS_*: the reduce-scatter instantiation (per-rank B shards, scattered rows)
// GEMM_*_NARROW: the float GEMM with an N = 64 tile (group 1 only, n <= 64; B
// maps with 64-column boxes)
enum GemmKind : int {
    GEMM_F16 = 0, GEMM_BF16 = 1, GEMM_INT_AS_F16 = 2, GEMM_RS_F16 = 3, GEMM_RS_BF16 = 4,
    GEMM_F16_NARROW = 5, GEMM_BF16_NARROW = 6
};
// group: 1 = one CTA per 128 x 256 tile, 2 = a CTA pair per 256 x 256 tile.
int gemm_group_for(int m);
// Work units (CTAs for group 1, CTA pairs for group 2) co-resident on the device;
// the persistent grid launches this many when a stream-K tail is used.
int gemm_units(GemmKind kind, int group, int num_sms);
// Stream-K partial slots reserved in the workspace: at most this many work units.
constexpr int kSkMaxUnits = 76;
cudaError_t launch_gemm(GemmKind kind, int group, const GemmParams &p, int num_sms, cudaStream_t stream);
int read_and_clear_gemm_status(int *status);
// Device address of the status word that bounded waits set to -7 (cached per device).
int *device_status_word();

// Id of the CUDA context current on this thread (cuCtxGetId: unique for the
// life of the process, so a context created after a device reset gets a new
// one), or 0 when there is none or it cannot be read.  Host-side state that
// belongs to a context (symbol addresses, function attributes) is cached
// under this id and looked up again when it changes; id 0 is never cached.
unsigned long long current_context_id();

// Records `msg` as this thread's mc2_last_error() text and returns `status`.
int record_error(int status, const char *msg);

cudaError_t launch_quant_pertoken(const ChunkPtrs &chunks, int rank_size, int64_t bs_local, int h, bool bf16,
                                  const void *smooth, __half *qh, int8_t *q_out, float *scale_out, void *comm_out,
                                  int num_sms, cudaStream_t stream);
// One launch doing both the per-token dynamic quant and the x2 widening
// (h % 8 == 0 and rank_size*h <= 32768, see a2a_prologue_fits).
bool a2a_prologue_fits(int rank_size, int64_t bs_local, int h);
cudaError_t launch_a2a_prologue(const ChunkPtrs &chunks, int rank_size, int64_t bs_local, int h, bool bf16,
                                const void *smooth, __half *qh, int8_t *q_out, float *scale_out, const int8_t *x2,
                                __half *x2h, int64_t x2_count, void *comm_out, int *status, uint64_t wait_limit_ns,
                                cudaStream_t stream);
cudaError_t launch_widen_i8(const int8_t *src, __half *dst, int64_t count, int num_sms, cudaStream_t stream);
// The full-quant path's widenings in one launch: each rank's int8 chunk to fp16
// in its own layout at dst_a + r*bs_local*h (h % 16 == 0), and x2 (x2_count
// elements, a multiple of 16) to dst_b; q_out (optional) receives the permuted
// int8 matrix.
cudaError_t launch_widen_a2a(const ChunkPtrs &chunks, int rank_size, int64_t bs_local, int h, __half *dst_a,
                             const int8_t *x2, __half *dst_b, int64_t x2_count, int8_t *q_out, int8_t *comm_out,
                             int num_sms, cudaStream_t stream);
cudaError_t launch_permute_widen_i8(const ChunkPtrs &chunks, int rank_size, int64_t bs_local, int h, __half *dst,
                                    int8_t *q_out, int8_t *comm_out, int num_sms, cudaStream_t stream);
// comm_out (optional, NULL for none): the received chunks stacked as
// (rank_size, bs_local, h) in their own dtype, written by the kernel that reads them.

// QuantAllReduce over `elems` elements (a multiple of 16) of each rank:
// x_kind 0 int8 / 1 e4m3fn / 2 e5m2; scale_kind 0 fp32 per 128 / 1 e8m0 per 32;
// out_kind 0 fp32 / 1 fp16 / 2 bf16; ranks 2, 4 or 8.
cudaError_t launch_quant_all_reduce(const void *const *x_chunks, const void *const *scale_chunks, int ranks,
                                    int64_t elems, int x_kind, int scale_kind, int out_kind, void *out, int num_sms,
                                    cudaStream_t stream);

}  // namespace mc2
