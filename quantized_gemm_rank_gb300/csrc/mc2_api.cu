// mc2_api.cu -- the C ABI declared in include/mc2_gb300.h: argument
// validation (constraints of "torch_npu.npu_all_gather_base_mm" 约束说明 and
// "aclnnAlltoAllQuantMatmul" 约束说明, plus this kernel's alignment needs),
// TMA tensor-map encoding, workspace carving and stream-ordered launches.
#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "gemm_tcgen05.cuh"
#include "internal.h"
#include "mc2_gb300.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return status;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ launch events
// The caller's events that mc2_set_launch_events installed on this thread:
// events[0] is recorded before a call's first kernel launch, events[i] after
// its i-th, on the call's stream.
constexpr int kMaxLaunchEvents = 8;
thread_local cudaEvent_t g_launch_events[kMaxLaunchEvents];
thread_local int g_num_launch_events = 0;

// Records the installed events of one call, in launch order.
class LaunchMarks {
  public:
    explicit LaunchMarks(cudaStream_t s) : s_(s) { mark(); }
    // after each kernel launch of the call
    void launched() { mark(); }

  private:
    void mark() {
        if (next_ < g_num_launch_events) cudaEventRecord(g_launch_events[next_], s_);
        ++next_;
    }
    cudaStream_t s_;
    int next_ = 0;
};

// One-shot test hook (mc2_test_expire_next_flag_waits): the wait limit the next
// AlltoAllQuantMatmul GEMM on this thread runs with, 0 when not armed.
thread_local uint64_t g_expire_next_flag_waits_ns = 0;

// ------------------------------------------------------------------ driver entry point
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_relaxed);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<EncodeTiledFn>(p);
            fn.store(f, std::memory_order_relaxed);
        }
    }
    return f;
}

// Encoded tensor maps, cached per host thread.  A map depends only on the base
// address, the sizes and the box, so a call that repeats an earlier call's
// buffers (the usual case in a serving or training loop) reuses the maps
// instead of encoding them again (cuTensorMapEncodeTiled is a host-side call
// of a fraction of a microsecond to a microsecond; an all-gather call encodes
// up to 11).  Direct-mapped: a key that hashes to an occupied slot replaces it.
struct MapKey {
    const void *base;
    uint64_t inner, outer;
    uint32_t box_inner, box_outer, groups;  // groups 0: a 2-D map
    bool operator==(const MapKey &o) const {
        return base == o.base && inner == o.inner && outer == o.outer && box_inner == o.box_inner &&
               box_outer == o.box_outer && groups == o.groups;
    }
};

constexpr int kMapCacheSlots = 64;
struct MapCacheSlot {
    MapKey key;
    CUtensorMap map;
    bool used;
};
thread_local MapCacheSlot g_map_cache[kMapCacheSlots];

MapCacheSlot &map_slot(const MapKey &k) {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    h ^= (k.inner * 0xC2B2AE3D27D4EB4Full) ^ (k.outer * 0x165667B19E3779F9ull);
    h ^= (static_cast<uint64_t>(k.box_inner) << 32 | k.box_outer) * 0x27D4EB2F165667C5ull + k.groups;
    h ^= h >> 29;
    return g_map_cache[h % kMapCacheSlots];
}

// 2-D map over a row-major (outer, inner) matrix with 16-bit elements and a
// 128-byte swizzle; out-of-range box elements read as zero.
bool make_map16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                uint32_t box_outer) {
    const MapKey key{base, inner, outer, box_inner, box_outer, 0};
    MapCacheSlot &slot = map_slot(key);
    if (slot.used && slot.key == key) {
        *m = slot.map;
        return true;
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    slot.key = key;
    slot.map = *m;
    slot.used = true;
    return true;
}

// N-major B (outer = k rows, inner = n columns, 16-bit) as a 3-D map
// [inner / 64][outer][64] (strides inner * 2 and 128 bytes), so one copy of box
// {64, box_outer, groups} brings `groups` 64-column slices, slice j landing
// 8 KiB after slice j - 1 (the layout of that many 2-D boxes).  Only for
// inner % 64 == 0: a partial last group would read into the next row.
bool make_map16_nmajor3d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_outer,
                         uint32_t groups) {
    if (inner % 64 != 0) return false;
    const MapKey key{base, inner, outer, 64, box_outer, groups};
    MapCacheSlot &slot = map_slot(key);
    if (slot.used && slot.key == key) {
        *m = slot.map;
        return true;
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, outer, inner / 64};
    cuuint64_t strides[2] = {inner * 2, 128};
    cuuint32_t box[3] = {64, box_outer, groups};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    slot.key = key;
    slot.map = *m;
    slot.used = true;
    return true;
}

struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
};

int current_device(DeviceInfo *info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    static std::atomic<int> sms_cache[64];
    int sms = dev < 64 ? sms_cache[dev].load(std::memory_order_relaxed) : 0;
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        if (major != 10 || minor != 3)
            return fail(MC2_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                        major, minor);
        if (dev < 64) sms_cache[dev].store(sms, std::memory_order_relaxed);
    }
    info->device = dev;
    info->num_sms = sms;
    return MC2_OK;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded device-side wait
constexpr int kKBlockTiles = 1024 / mc2::kBK;      // k-tiles per exact fp32 K block (1024 * 127^2 < 2^24)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct A2AWorkspace {
    size_t x2h = 0, ah = 0, scale = 0, sk_partials = 0, sk_flags = 0, total = 0;
    int num_tiles = 0, nkb = 0, sk_slots = 0;
};

// Workspace: x2 widened (K, N) fp16 | activations as fp16 (BS/R, K) | scales |
// stream-K partial slots (2 x 128 x 256 int32 each) | stream-K flags (2 per tile,
// 8 bytes each, never zeroed: they carry the launch's epoch).
A2AWorkspace a2a_layout(int rank_size, int64_t bs_local, int64_t h, int64_t n) {
    A2AWorkspace w;
    const size_t K = static_cast<size_t>(rank_size) * static_cast<size_t>(h);
    const int group = mc2::gemm_group_for(static_cast<int>(bs_local));
    const int64_t tile_m = static_cast<int64_t>(mc2::kBM) * group;
    w.num_tiles = static_cast<int>(((bs_local + tile_m - 1) / tile_m) * ((n + mc2::kBN - 1) / mc2::kBN));
    const int64_t num_k = (static_cast<int64_t>(K) + mc2::kBK - 1) / mc2::kBK;
    w.nkb = static_cast<int>((num_k + kKBlockTiles - 1) / kKBlockTiles);
    const int64_t blocks = static_cast<int64_t>(w.num_tiles) * w.nkb;
    // a writer uses the slot of its work unit, so a tail needs one slot per unit
    // (kSkMaxUnits on GB300); problems with fewer K blocks than that reserve none
    w.sk_slots = blocks >= mc2::kSkMaxUnits ? mc2::kSkMaxUnits : 0;
    w.x2h = 0;
    w.ah = align_up(w.x2h + K * static_cast<size_t>(n) * 2, 256);
    w.scale = align_up(w.ah + static_cast<size_t>(bs_local) * K * 2, 256);
    w.sk_partials = align_up(w.scale + static_cast<size_t>(bs_local) * 4, 256);
    w.sk_flags = align_up(w.sk_partials + static_cast<size_t>(w.sk_slots) * 2 * mc2::kBM * mc2::kBN * 4, 256);
    w.total = align_up(w.sk_flags + static_cast<size_t>(w.num_tiles) * 2 * 8, 256);
    return w;
}

int validate_a2a(int rank_size, int64_t bs_local, int64_t h, int64_t n, int x1_quant_mode, int x1_dtype) {
    if (rank_size != 2 && rank_size != 4 && rank_size != 8)
        return fail(MC2_ERR_SHAPE, "rank_size must be 2, 4 or 8 (got %d)", rank_size);
    if (bs_local < 1 || h < 1 || n < 1)
        return fail(MC2_ERR_SHAPE, "empty tensors are not supported (bs_local=%lld h=%lld n=%lld)",
                    (long long)bs_local, (long long)h, (long long)n);
    if (bs_local * rank_size > INT32_MAX) return fail(MC2_ERR_SHAPE, "BS = rank_size*bs_local exceeds INT32_MAX");
    if (n > INT32_MAX) return fail(MC2_ERR_SHAPE, "N exceeds INT32_MAX");
    const int64_t K = static_cast<int64_t>(rank_size) * h;
    if (K > 35000) return fail(MC2_ERR_SHAPE, "rank_size*H = %lld is outside [1, 35000]", (long long)K);
    if (K % 16 != 0) return fail(MC2_ERR_SHAPE, "rank_size*H = %lld is not a multiple of 16", (long long)K);
    if (x1_quant_mode == MC2_QUANT_PERTOKEN_DYNAMIC) {
        if (x1_dtype != MC2_BF16 && x1_dtype != MC2_F16)
            return fail(MC2_ERR_DTYPE, "x1QuantMode 7 needs bf16 or fp16 chunks (got dtype %d)", x1_dtype);
    } else if (x1_quant_mode == MC2_QUANT_PERTOKEN) {
        if (x1_dtype != MC2_I8) return fail(MC2_ERR_DTYPE, "x1QuantMode 3 needs int8 chunks (got dtype %d)", x1_dtype);
    } else {
        return fail(MC2_ERR_DTYPE, "x1QuantMode must be 3 (pertoken) or 7 (pertoken dynamic), got %d", x1_quant_mode);
    }
    if (n % 16 != 0) return fail(MC2_ERR_UNSUPPORTED, "this kernel needs N %% 16 == 0 (got %lld)", (long long)n);
    return MC2_OK;
}

}  // namespace

namespace mc2 {
int record_error(int status, const char *msg) { return fail(status, "%s", msg); }
}  // namespace mc2

extern "C" {

const char *mc2_status_str(int status) {
    switch (status) {
        case MC2_OK: return "MC2_OK";
        case MC2_ERR_NULL: return "MC2_ERR_NULL";
        case MC2_ERR_SHAPE: return "MC2_ERR_SHAPE";
        case MC2_ERR_DTYPE: return "MC2_ERR_DTYPE";
        case MC2_ERR_UNSUPPORTED: return "MC2_ERR_UNSUPPORTED";
        case MC2_ERR_WORKSPACE: return "MC2_ERR_WORKSPACE";
        case MC2_ERR_CUDA: return "MC2_ERR_CUDA";
        case MC2_ERR_TIMEOUT: return "MC2_ERR_TIMEOUT";
    }
    return "MC2_ERR_UNKNOWN";
}

const char *mc2_last_error(void) { return g_last_error; }

int mc2_device_status(void) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    int st = 0;
    if (mc2::read_and_clear_gemm_status(&st) != 0) return fail(MC2_ERR_CUDA, "reading the device status word failed");
    if (st != 0) return fail(MC2_ERR_TIMEOUT, "a bounded wait inside the GEMM kernel gave up");
    return MC2_OK;
}

int mc2_set_launch_events(void *const *events, int count) {
    g_last_error[0] = '\0';
    if (count < 0 || count > kMaxLaunchEvents)
        return fail(MC2_ERR_SHAPE, "count must be in [0, %d] (got %d)", kMaxLaunchEvents, count);
    if (count > 0 && !events) return fail(MC2_ERR_NULL, "events is NULL");
    for (int i = 0; i < count; ++i)
        if (!events[i]) return fail(MC2_ERR_NULL, "events[%d] is NULL", i);
    for (int i = 0; i < count; ++i) g_launch_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_num_launch_events = count;
    return MC2_OK;
}

int mc2_test_expire_next_flag_waits(uint64_t wait_limit_ns) {
    g_last_error[0] = '\0';
    if (wait_limit_ns == 0 || wait_limit_ns > kWaitLimitNs)
        return fail(MC2_ERR_SHAPE, "wait_limit_ns must be in [1, %llu] (got %llu)", (unsigned long long)kWaitLimitNs,
                    (unsigned long long)wait_limit_ns);
    g_expire_next_flag_waits_ns = wait_limit_ns;
    return MC2_OK;
}

int mc2_all_gather_mm(const void *const *x_chunks, int world_size, int64_t m_local, int64_t k, const void *x2,
                      int64_t n, int x2_is_nk, const void *bias, int dtype, int gather_output, void *out,
                      void *gathered, void *stream) {
    g_last_error[0] = '\0';
    if (!x_chunks) return fail(MC2_ERR_NULL, "x_chunks is NULL");
    if (!x2) return fail(MC2_ERR_NULL, "x2 is NULL");
    if (!out) return fail(MC2_ERR_NULL, "out is NULL");
    if (world_size != 2 && world_size != 4 && world_size != 8)
        return fail(MC2_ERR_SHAPE, "world_size must be 2, 4 or 8 (got %d)", world_size);
    for (int r = 0; r < world_size; ++r)
        if (!x_chunks[r]) return fail(MC2_ERR_NULL, "x_chunks[%d] is NULL", r);
    if (dtype != MC2_F16 && dtype != MC2_BF16)
        return fail(MC2_ERR_DTYPE, "dtype must be MC2_F16 or MC2_BF16 (got %d)", dtype);
    if (m_local < 1 || n < 1)
        return fail(MC2_ERR_SHAPE, "empty tensors are not supported (m_local=%lld n=%lld)", (long long)m_local,
                    (long long)n);
    if (k < 256 || k >= 65535) return fail(MC2_ERR_SHAPE, "k must be in [256, 65535) (got %lld)", (long long)k);
    if (gather_output && !gathered) return fail(MC2_ERR_NULL, "gather_output is set but gathered is NULL");
    if (!gather_output && gathered) return fail(MC2_ERR_SHAPE, "gathered must be NULL when gather_output is 0");
    const int64_t m = m_local * world_size;
    if (m > INT32_MAX || n > INT32_MAX) return fail(MC2_ERR_SHAPE, "m or n exceeds INT32_MAX");
    if (m_local % 8 != 0)
        return fail(MC2_ERR_UNSUPPORTED, "this kernel needs m_local %% 8 == 0 (got %lld)", (long long)m_local);
    if (k % 8 != 0 || n % 8 != 0)
        return fail(MC2_ERR_UNSUPPORTED, "this kernel needs k %% 8 == 0 and n %% 8 == 0 (k=%lld n=%lld)",
                    (long long)k, (long long)n);
    for (int r = 0; r < world_size; ++r)
        if (!aligned16(x_chunks[r])) return fail(MC2_ERR_UNSUPPORTED, "x_chunks[%d] is not 16-byte aligned", r);
    if (!aligned16(x2) || !aligned16(out) || (bias && !aligned16(bias)) || (gathered && !aligned16(gathered)))
        return fail(MC2_ERR_UNSUPPORTED, "x2, out, bias and gathered must be 16-byte aligned");

    DeviceInfo dev;
    if (int st = current_device(&dev)) return st;

    mc2::GemmParams p;
    memset(&p, 0, sizeof(p));
    // A: one map per rank's chunk, box rows = the largest power of two dividing
    // both m_local and the 128-row tile, so that no box crosses a chunk.  When the
    // chunks lie back to back (the slices of one receive buffer, as an all-gather
    // writes them) and a chunk is shorter than a tile, A is read through one map of
    // the whole (m, k) instead: one 128-row box per k-tile rather than one small box
    // per chunk (on 8 chunks of 16 rows that is 8 copies instead of 64 for a K of 512).
    int box_rows = mc2::kBM;
    while (m_local % box_rows != 0) box_rows >>= 1;
    bool back_to_back = true;
    const int64_t chunk_bytes = m_local * k * 2;
    for (int r = 1; r < world_size; ++r)
        if (static_cast<const char *>(x_chunks[r]) != static_cast<const char *>(x_chunks[0]) + r * chunk_bytes)
            back_to_back = false;
    if (back_to_back && box_rows < mc2::kBM) {
        if (!make_map16(&p.a_maps[0], x_chunks[0], k, m, mc2::kBK, mc2::kBM))
            return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for the chunks (one buffer)");
        p.num_a_maps = 1;
        p.a_mode = mc2::A_SINGLE;
    } else {
        for (int r = 0; r < world_size; ++r)
            if (!make_map16(&p.a_maps[r], x_chunks[r], k, m_local, mc2::kBK, box_rows))
                return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for x_chunks[%d]", r);
        p.num_a_maps = world_size;
        p.a_mode = mc2::A_MCONCAT;
        p.a_box_rows = box_rows;
    }
    p.m_local = static_cast<int>(m_local);
    const int group = mc2::gemm_group_for(static_cast<int>(m));
    // one CTA and an output at most 64 wide: the narrow tile (N = 64), whose short
    // stages let the whole K of such a problem be in flight at once
    const bool narrow = group == 1 && n <= 64;
    const uint32_t b_cols = narrow ? 64u : static_cast<uint32_t>(mc2::kBN / group);   // B columns per CTA
    if (x2_is_nk) {
        if (!make_map16(&p.b_map, x2, k, n, mc2::kBK, b_cols))
            return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for x2 (n, k)");
        p.b_mn_major = 0;
    } else {
        if (make_map16_nmajor3d(&p.b_map, x2, n, k, mc2::kBK, b_cols / 64))
            p.b_3d = 1;
        else if (!make_map16(&p.b_map, x2, n, k, 64, mc2::kBK))
            return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for x2 (k, n)");
        p.b_mn_major = 1;
    }
    if (gather_output) {
        if (!make_map16(&p.g_map, gathered, k, m, mc2::kBK, mc2::kBM))
            return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for gathered");
        p.gather = 1;
    }
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.kblock_tiles = kKBlockTiles;
    p.out = out;
    if (!make_map16(&p.out_map, p.out, static_cast<uint64_t>(p.n), static_cast<uint64_t>(p.m), 64, 32))
        return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for the output");
    p.bias16 = bias;
    p.wait_limit_ns = kWaitLimitNs;
    const mc2::GemmKind kind = narrow ? (dtype == MC2_BF16 ? mc2::GEMM_BF16_NARROW : mc2::GEMM_F16_NARROW)
                                      : (dtype == MC2_BF16 ? mc2::GEMM_BF16 : mc2::GEMM_F16);
    LaunchMarks marks(static_cast<cudaStream_t>(stream));
    cudaError_t e = mc2::launch_gemm(kind, group, p, dev.num_sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    marks.launched();
    return MC2_OK;
}

int mc2_matmul_reduce_scatter(const void *const *x_chunks, const void *const *w_chunks, int world_size, int64_t m,
                              int64_t k_local, int64_t n, int w_is_nk, const void *bias, int dtype,
                              void *const *out_chunks, void *stream) {
    g_last_error[0] = '\0';
    if (!x_chunks || !w_chunks || !out_chunks) return fail(MC2_ERR_NULL, "x_chunks, w_chunks and out_chunks are required");
    if (world_size != 2 && world_size != 4 && world_size != 8)
        return fail(MC2_ERR_SHAPE, "world_size must be 2, 4 or 8 (got %d)", world_size);
    for (int r = 0; r < world_size; ++r)
        if (!x_chunks[r] || !w_chunks[r] || !out_chunks[r])
            return fail(MC2_ERR_NULL, "x_chunks[%d], w_chunks[%d] or out_chunks[%d] is NULL", r, r, r);
    if (dtype != MC2_F16 && dtype != MC2_BF16)
        return fail(MC2_ERR_DTYPE, "dtype must be MC2_F16 or MC2_BF16 (got %d)", dtype);
    if (m < 1 || n < 1) return fail(MC2_ERR_SHAPE, "empty tensors are not supported (m=%lld n=%lld)", (long long)m,
                                    (long long)n);
    if (m % world_size != 0)
        return fail(MC2_ERR_SHAPE, "m = %lld is not divisible by world_size %d (the scatter splits m)", (long long)m,
                    world_size);
    if (k_local < 256 || k_local >= 65535)
        return fail(MC2_ERR_SHAPE, "the contraction size k must be in [256, 65535) (got %lld)", (long long)k_local);
    if (m > INT32_MAX || n > INT32_MAX) return fail(MC2_ERR_SHAPE, "m or n exceeds INT32_MAX");
    if (k_local % mc2::kBK != 0)
        return fail(MC2_ERR_UNSUPPORTED, "this kernel needs k %% 64 == 0 (a k-tile may not straddle two ranks), got %lld",
                    (long long)k_local);
    if (n % 8 != 0) return fail(MC2_ERR_UNSUPPORTED, "this kernel needs n %% 8 == 0 (got %lld)", (long long)n);
    for (int r = 0; r < world_size; ++r)
        if (!aligned16(x_chunks[r]) || !aligned16(w_chunks[r]) || !aligned16(out_chunks[r]))
            return fail(MC2_ERR_UNSUPPORTED, "rank %d's buffers must be 16-byte aligned", r);
    if (bias && !aligned16(bias)) return fail(MC2_ERR_UNSUPPORTED, "bias must be 16-byte aligned");

    DeviceInfo dev;
    if (int st = current_device(&dev)) return st;
    mc2::GemmParams p;
    memset(&p, 0, sizeof(p));
    const int group = mc2::gemm_group_for(static_cast<int>(m));
    // A: rank r's activations X_r (m, k_local) are k-slice r of the contraction;
    // B: rank r's weight shard, w (n, k_local) K-major or x2 (k_local, n) N-major
    for (int r = 0; r < world_size; ++r) {
        if (!make_map16(&p.a_maps[r], x_chunks[r], k_local, m, mc2::kBK, mc2::kBM))
            return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for x_chunks[%d]", r);
        const bool okb = w_is_nk ? make_map16(&p.b_rank_maps[r], w_chunks[r], k_local, n, mc2::kBK, mc2::kBN / group)
                                 : make_map16(&p.b_rank_maps[r], w_chunks[r], n, k_local, 64, mc2::kBK);
        if (!okb) return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for w_chunks[%d]", r);
        p.out_chunks[r] = out_chunks[r];
    }
    p.num_a_maps = world_size;
    p.a_mode = mc2::A_KINTERLEAVE;
    p.k_local = static_cast<int>(k_local);
    p.b_mn_major = w_is_nk ? 0 : 1;
    p.out_rows = static_cast<int>(m / world_size);
    // a warp's 32 output rows belong to one rank when out_rows % 32 == 0: the
    // epilogue then stores through one tensor map per rank's output
    if (p.out_rows % 32 == 0) {
        for (int r = 0; r < world_size; ++r)
            if (!make_map16(&p.out_rank_maps[r], out_chunks[r], static_cast<uint64_t>(n),
                            static_cast<uint64_t>(p.out_rows), 64, 32))
                return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for out_chunks[%d]", r);
        p.rs_tma = 1;
    }
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k_local * world_size);
    p.kblock_tiles = kKBlockTiles;
    p.bias16 = bias;
    p.wait_limit_ns = kWaitLimitNs;
    LaunchMarks marks(static_cast<cudaStream_t>(stream));
    cudaError_t e = mc2::launch_gemm(dtype == MC2_BF16 ? mc2::GEMM_RS_BF16 : mc2::GEMM_RS_F16, group, p, dev.num_sms,
                                     static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    marks.launched();
    return MC2_OK;
}

int mc2_matmul_weight_grad(const void *dy, int64_t m, int64_t n, const void *x, int64_t k, int dtype, void *dw,
                           void *db, void *stream) {
    g_last_error[0] = '\0';
    if (!dy || !x || !dw) return fail(MC2_ERR_NULL, "dy, x and dw are required");
    if (dtype != MC2_F16 && dtype != MC2_BF16)
        return fail(MC2_ERR_DTYPE, "dtype must be MC2_F16 or MC2_BF16 (got %d)", dtype);
    if (m < 1 || n < 1 || k < 1)
        return fail(MC2_ERR_SHAPE, "empty tensors are not supported (m=%lld n=%lld k=%lld)", (long long)m,
                    (long long)n, (long long)k);
    if (m > INT32_MAX || n > INT32_MAX || k > INT32_MAX) return fail(MC2_ERR_SHAPE, "m, n or k exceeds INT32_MAX");
    if (n % 8 != 0 || k % 8 != 0)
        return fail(MC2_ERR_UNSUPPORTED, "this kernel needs n %% 8 == 0 and k %% 8 == 0 (got n=%lld k=%lld)",
                    (long long)n, (long long)k);
    if (!aligned16(dy) || !aligned16(x) || !aligned16(dw) || (db && !aligned16(db)))
        return fail(MC2_ERR_UNSUPPORTED, "all tensors must be 16-byte aligned");

    DeviceInfo dev;
    if (int st = current_device(&dev)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    LaunchMarks marks(s);
    // dW (n, k) = dY^T @ X: A = dY^T read M-major from dY (m, n), B = X (m, k) N-major,
    // the contraction runs down the m rows of both; the same launch sums A's rows
    // over the contraction (the column sums of dY) into db
    mc2::GemmParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map16(&p.a_maps[0], dy, n, m, 64, mc2::kBK)) return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for dy");
    const int wgroup = mc2::gemm_group_for(static_cast<int>(n));
    if (make_map16_nmajor3d(&p.b_map, x, k, m, mc2::kBK, (mc2::kBN / wgroup) / 64))
        p.b_3d = 1;
    else if (!make_map16(&p.b_map, x, k, m, 64, mc2::kBK))
        return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for x");
    p.num_a_maps = 1;
    p.a_mode = mc2::A_SINGLE_MN;
    p.b_mn_major = 1;
    p.m = static_cast<int>(n);
    p.n = static_cast<int>(k);
    p.k = static_cast<int>(m);
    p.kblock_tiles = kKBlockTiles;
    p.out = dw;
    if (!make_map16(&p.out_map, p.out, static_cast<uint64_t>(p.n), static_cast<uint64_t>(p.m), 64, 32))
        return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for the output");
    p.colsum_out = db;
    p.wait_limit_ns = kWaitLimitNs;
    const int group = mc2::gemm_group_for(static_cast<int>(n));
    e = mc2::launch_gemm(dtype == MC2_BF16 ? mc2::GEMM_BF16 : mc2::GEMM_F16, group, p, dev.num_sms, s);
    if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    marks.launched();
    return MC2_OK;
}

int mc2_quant_all_reduce(const void *const *x_chunks, const void *const *scale_chunks, int world_size, int64_t bs,
                         int64_t h, int x_dtype, int scale_dtype, int out_dtype, void *out, void *stream) {
    g_last_error[0] = '\0';
    if (!x_chunks || !scale_chunks || !out) return fail(MC2_ERR_NULL, "x_chunks, scale_chunks and out are required");
    if (world_size != 2 && world_size != 4 && world_size != 8)
        return fail(MC2_ERR_SHAPE, "world_size must be 2, 4 or 8 (got %d)", world_size);
    for (int r = 0; r < world_size; ++r)
        if (!x_chunks[r] || !scale_chunks[r]) return fail(MC2_ERR_NULL, "x_chunks[%d] or scale_chunks[%d] is NULL", r, r);
    if (bs < 1) return fail(MC2_ERR_SHAPE, "empty tensors are not supported (bs=%lld)", (long long)bs);
    if (h < 1024 || h > 8192 || h % 128 != 0)
        return fail(MC2_ERR_SHAPE, "H must be a multiple of 128 in [1024, 8192] (got %lld)", (long long)h);
    if (x_dtype != MC2_I8 && x_dtype != MC2_F8E4M3 && x_dtype != MC2_F8E5M2)
        return fail(MC2_ERR_DTYPE, "x must be MC2_I8, MC2_F8E4M3 or MC2_F8E5M2 (got %d)", x_dtype);
    if (scale_dtype != MC2_F32 && scale_dtype != MC2_E8M0)
        return fail(MC2_ERR_DTYPE, "scales must be MC2_F32 or MC2_E8M0 (got %d)", scale_dtype);
    if (scale_dtype == MC2_E8M0 && x_dtype == MC2_I8)
        return fail(MC2_ERR_DTYPE, "e8m0 (mx) scales need fp8 x (MC2_F8E4M3 or MC2_F8E5M2)");
    if (out_dtype != MC2_F32 && out_dtype != MC2_F16 && out_dtype != MC2_BF16)
        return fail(MC2_ERR_DTYPE, "out must be MC2_F32, MC2_F16 or MC2_BF16 (got %d)", out_dtype);
    if (bs > INT64_MAX / 8192) return fail(MC2_ERR_SHAPE, "bs too large");
    for (int r = 0; r < world_size; ++r)
        if (!aligned16(x_chunks[r]) || !aligned16(scale_chunks[r]))
            return fail(MC2_ERR_UNSUPPORTED, "x_chunks[%d] and scale_chunks[%d] must be 16-byte aligned", r, r);
    if (!aligned16(out)) return fail(MC2_ERR_UNSUPPORTED, "out must be 16-byte aligned");

    DeviceInfo dev;
    if (int st = current_device(&dev)) return st;
    const int x_kind = x_dtype == MC2_I8 ? 0 : (x_dtype == MC2_F8E4M3 ? 1 : 2);
    const int out_kind = out_dtype == MC2_F32 ? 0 : (out_dtype == MC2_F16 ? 1 : 2);
    LaunchMarks marks(static_cast<cudaStream_t>(stream));
    cudaError_t e = mc2::launch_quant_all_reduce(x_chunks, scale_chunks, world_size, bs * h, x_kind,
                                                 scale_dtype == MC2_E8M0 ? 1 : 0, out_kind, out, dev.num_sms,
                                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "QuantAllReduce launch: %s", cudaGetErrorString(e));
    marks.launched();
    return MC2_OK;
}

int mc2_alltoall_quant_mm_workspace(int rank_size, int64_t bs_local, int64_t h, int64_t n, int x1_quant_mode,
                                    int x1_dtype, size_t *bytes) {
    g_last_error[0] = '\0';
    if (!bytes) return fail(MC2_ERR_NULL, "bytes is NULL");
    if (int st = validate_a2a(rank_size, bs_local, h, n, x1_quant_mode, x1_dtype)) return st;
    *bytes = a2a_layout(rank_size, bs_local, h, n).total;
    return MC2_OK;
}

int mc2_alltoall_quant_mm(const void *const *chunks, int rank_size, int64_t bs_local, int64_t h, int x1_dtype,
                          const void *x1_scale, const int8_t *x2, const float *x2_scale, const void *bias,
                          int bias_dtype, int x1_quant_mode, int x2_quant_mode, int64_t n, void *out,
                          void *alltoall_out, int8_t *q_out, float *x1_scale_out, int32_t *acc_out, void *workspace,
                          size_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    if (!chunks) return fail(MC2_ERR_NULL, "chunks is NULL");
    if (!x2) return fail(MC2_ERR_NULL, "x2 is NULL");
    if (!x2_scale) return fail(MC2_ERR_NULL, "x2_scale is NULL");
    if (!out) return fail(MC2_ERR_NULL, "output is NULL");
    if (!bias) return fail(MC2_ERR_NULL, "bias is NULL (biasOptional may not be NULL on this op)");
    if (int st = validate_a2a(rank_size, bs_local, h, n, x1_quant_mode, x1_dtype)) return st;
    for (int r = 0; r < rank_size; ++r)
        if (!chunks[r]) return fail(MC2_ERR_NULL, "chunks[%d] is NULL", r);
    if (x2_quant_mode != MC2_QUANT_PERCHANNEL)
        return fail(MC2_ERR_DTYPE, "x2QuantMode must be 2 (perchannel), got %d", x2_quant_mode);
    if (bias_dtype != MC2_F32 && bias_dtype != MC2_BF16)
        return fail(MC2_ERR_DTYPE, "bias dtype must be MC2_F32 or MC2_BF16 (got %d)", bias_dtype);
    if (x1_quant_mode == MC2_QUANT_PERTOKEN && !x1_scale)
        return fail(MC2_ERR_NULL, "x1QuantMode 3 needs the per-token x1 scale");
    for (int r = 0; r < rank_size; ++r)
        if (!aligned16(chunks[r])) return fail(MC2_ERR_UNSUPPORTED, "chunks[%d] is not 16-byte aligned", r);
    if (!aligned16(x2) || !aligned16(out) || !aligned16(x2_scale) || !aligned16(bias) ||
        (x1_scale && !aligned16(x1_scale)) || (q_out && !aligned16(q_out)) || (acc_out && !aligned16(acc_out)) ||
        (x1_scale_out && !aligned16(x1_scale_out)) || (alltoall_out && !aligned16(alltoall_out)))
        return fail(MC2_ERR_UNSUPPORTED, "all tensors must be 16-byte aligned");
    const A2AWorkspace ws = a2a_layout(rank_size, bs_local, h, n);
    if (!workspace || workspace_bytes < ws.total)
        return fail(MC2_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", ws.total,
                    workspace ? workspace_bytes : (size_t)0);
    if (!aligned16(workspace)) return fail(MC2_ERR_UNSUPPORTED, "workspace must be 16-byte aligned");

    DeviceInfo dev;
    if (int st = current_device(&dev)) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    __half *x2h = reinterpret_cast<__half *>(wsb + ws.x2h);
    __half *ah = reinterpret_cast<__half *>(wsb + ws.ah);
    float *scale = x1_scale_out ? x1_scale_out : reinterpret_cast<float *>(wsb + ws.scale);
    const int64_t K = static_cast<int64_t>(rank_size) * h;
    mc2::ChunkPtrs cp;
    memset(&cp, 0, sizeof(cp));
    for (int r = 0; r < rank_size; ++r) cp.p[r] = chunks[r];

    // Mode 3 with h % 64 == 0: each chunk is widened in place of its own (with x2,
    // in one pass) and the GEMM reads the permuted matrix through one tensor map
    // per chunk (a k-tile never straddles two chunks); otherwise the widening
    // writes it permuted.
    const bool a_by_chunk = x1_quant_mode == MC2_QUANT_PERTOKEN && h % mc2::kBK == 0;
    // stream-K tail: the tiles left over after whole waves of the co-resident pairs
    // (or CTAs) are split by K blocks over all of them (needs >= 2 K blocks a tile)
    const int group = mc2::gemm_group_for(static_cast<int>(bs_local));
    const int units = mc2::gemm_units(mc2::GEMM_INT_AS_F16, group, dev.num_sms);
    int sk_tiles = 0;
    if (ws.nkb >= 2 && units <= ws.sk_slots && ws.num_tiles % units != 0) sk_tiles = ws.num_tiles % units;
    cudaError_t e = cudaSuccess;
    bool x2_done = false;
    if (x1_quant_mode == MC2_QUANT_PERTOKEN && x1_scale_out) {
        // mode 3: the per-token scales are the caller's; x1_scale_out receives a copy
        e = cudaMemcpyAsync(x1_scale_out, x1_scale, static_cast<size_t>(bs_local) * 4, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "x1 scale copy: %s", cudaGetErrorString(e));
    }
    LaunchMarks marks(s);
    if (x1_quant_mode == MC2_QUANT_PERTOKEN_DYNAMIC && mc2::a2a_prologue_fits(rank_size, bs_local, static_cast<int>(h))) {
        e = mc2::launch_a2a_prologue(cp, rank_size, bs_local, static_cast<int>(h), x1_dtype == MC2_BF16, x1_scale, ah,
                                     q_out, scale, x2, x2h, K * n, alltoall_out,
                                     mc2::device_status_word(), kWaitLimitNs, s);
        x2_done = true;
    } else if (x1_quant_mode == MC2_QUANT_PERTOKEN_DYNAMIC) {
        e = mc2::launch_quant_pertoken(cp, rank_size, bs_local, static_cast<int>(h), x1_dtype == MC2_BF16, x1_scale,
                                       ah, q_out, scale, alltoall_out, dev.num_sms, s);
    } else {
        // mode 3: the scales are the caller's; the int8 chunks and x2 are widened, in
        // one pass when the GEMM reads the chunks in their own layout
        if (a_by_chunk) {
            e = mc2::launch_widen_a2a(cp, rank_size, bs_local, static_cast<int>(h), ah, x2, x2h, K * n, q_out,
                                      static_cast<int8_t *>(alltoall_out), dev.num_sms, s);
            x2_done = true;
        } else
            e = mc2::launch_permute_widen_i8(cp, rank_size, bs_local, static_cast<int>(h), ah, q_out,
                                             static_cast<int8_t *>(alltoall_out), dev.num_sms, s);
        scale = const_cast<float *>(static_cast<const float *>(x1_scale));
    }
    if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "prologue launch: %s", cudaGetErrorString(e));
    marks.launched();
    if (!x2_done) {
        e = mc2::launch_widen_i8(x2, x2h, K * n, dev.num_sms, s);
        if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "x2 widening launch: %s", cudaGetErrorString(e));
        marks.launched();
    }

    mc2::GemmParams p;
    memset(&p, 0, sizeof(p));
    if (a_by_chunk) {
        for (int r = 0; r < rank_size; ++r)
            if (!make_map16(&p.a_maps[r], ah + static_cast<size_t>(r) * bs_local * h, h, bs_local, mc2::kBK, mc2::kBM))
                return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for widened chunk %d", r);
    } else if (!make_map16(&p.a_maps[0], ah, K, bs_local, mc2::kBK, mc2::kBM)) {
        return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for the quantised activations");
    }
    if (make_map16_nmajor3d(&p.b_map, x2h, n, K, mc2::kBK, (mc2::kBN / group) / 64))
        p.b_3d = 1;
    else if (!make_map16(&p.b_map, x2h, n, K, 64, mc2::kBK))
        return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for x2");
    p.num_a_maps = a_by_chunk ? rank_size : 1;
    p.a_mode = a_by_chunk ? mc2::A_KINTERLEAVE : mc2::A_SINGLE;
    p.k_local = static_cast<int>(h);
    p.b_mn_major = 1;
    p.m = static_cast<int>(bs_local);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(K);
    p.kblock_tiles = kKBlockTiles;
    p.out = out;
    if (!make_map16(&p.out_map, p.out, static_cast<uint64_t>(p.n), static_cast<uint64_t>(p.m), 64, 32))
        return fail(MC2_ERR_CUDA, "cuTensorMapEncodeTiled failed for the output");
    p.x1_scale = scale;
    p.x2_scale = x2_scale;
    p.bias_q = bias;
    p.bias_q_bf16 = bias_dtype == MC2_BF16;
    p.acc_out = acc_out;
    p.sk_tiles = sk_tiles;
    p.sk_partials = reinterpret_cast<int32_t *>(wsb + ws.sk_partials);
    p.sk_flags = reinterpret_cast<unsigned long long *>(wsb + ws.sk_flags);
    p.wait_limit_ns = kWaitLimitNs;
    if (g_expire_next_flag_waits_ns != 0) {
        // the test hook: this launch's FINISH parts expect one writer too many
        p.wait_limit_ns = g_expire_next_flag_waits_ns;
        p.sk_extra_writers = 1;
        g_expire_next_flag_waits_ns = 0;
    }
    e = mc2::launch_gemm(mc2::GEMM_INT_AS_F16, group, p, dev.num_sms, s);
    if (e != cudaSuccess) return fail(MC2_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    marks.launched();
    return MC2_OK;
}

}  // extern "C"
