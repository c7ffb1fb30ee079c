// gemm_kernels.cu -- instantiations and launch of the fused MC2 GEMM.
#include <atomic>
#include <chrono>
#include "gemm_tcgen05.cuh"
#include "internal.h"

namespace mc2 {

__device__ int g_gemm_status = 0;

unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static std::atomic<GetCurrentFn> get_current{nullptr};
    static std::atomic<GetIdFn> get_id{nullptr};
    GetCurrentFn gc = get_current.load(std::memory_order_relaxed);
    GetIdFn gi = get_id.load(std::memory_order_relaxed);
    if (!gc || !gi) {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
            qa != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
            qb != cudaDriverEntryPointSuccess)
            return 0;
        gc = reinterpret_cast<GetCurrentFn>(a);
        gi = reinterpret_cast<GetIdFn>(b);
        get_current.store(gc, std::memory_order_relaxed);
        get_id.store(gi, std::memory_order_relaxed);
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (gc(&ctx) != CUDA_SUCCESS || ctx == nullptr || gi(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

namespace {

// CTA pairs of this instantiation that fit on the device at once, from the
// occupancy calculator (cached per device).
template <bool kBF16, bool kIntPath, bool kRS = false>
int concurrent_pairs(int num_sms) {
    using Cfg = TileCfg<2, true>;
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return num_sms / 2;
    int clusters = dev < 64 ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (clusters == 0) {
        auto kern = mc2_gemm_kernel<2, kBF16, kIntPath, kRS>;
        // without the opt-in the occupancy query below fails and the fallback applies
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes) != cudaSuccess)
            return num_sms / 2;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.blockDim = dim3(kNumThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;
        cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1)
            clusters = num_sms / 2;
        if (dev < 64) cached[dev].store(clusters, std::memory_order_relaxed);
    }
    return clusters;
}

// Epochs of the stream-K flags: consecutive per launch from a per-process
// starting point (clock and address mixed), in [2^20, 2^40), far from the
// small integers a fresh buffer may hold and from another process's epochs.
unsigned long long sk_epoch_seed() {
    static int anchor;
    unsigned long long x = static_cast<unsigned long long>(
                               std::chrono::steady_clock::now().time_since_epoch().count()) ^
                           reinterpret_cast<uintptr_t>(&anchor);
    x ^= x >> 33;
    x *= 0xff51afd7ed558ccdull;
    x ^= x >> 33;
    return x;
}

unsigned long long next_sk_epoch() {
    static std::atomic<unsigned long long> counter{sk_epoch_seed()};
    constexpr unsigned long long kLo = 1ull << 20, kSpan = (1ull << 40) - (1ull << 20);
    return kLo + counter.fetch_add(1, std::memory_order_relaxed) % kSpan;
}

template <int kG, bool kBF16, bool kIntPath, bool kRS = false, bool kDyn = false, bool kNarrow = false>
cudaError_t launch_one(const GemmParams &p_in, int num_sms, cudaStream_t stream) {
    using Cfg = TileCfg<kG, true, kNarrow>;
    auto kern = mc2_gemm_kernel<kG, kBF16, kIntPath, kRS, kDyn, kNarrow>;
    GemmParams p = p_in;
    // once per host thread and context (a device switch or reset makes a new
    // context): the status word's address and the shared-memory opt-in
    thread_local unsigned long long ready_ctx = 0;
    thread_local int *status_word = nullptr;
    const unsigned long long ctx = current_context_id();
    cudaError_t e = cudaSuccess;
    if (ctx == 0 || ctx != ready_ctx) {
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status_word), g_gemm_status);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        ready_ctx = ctx;
    }
    p.status = status_word;
    const int num_tiles = ((p.m + Cfg::kTileM - 1) / Cfg::kTileM) * ((p.n + kBN - 1) / kBN);
    // stream-K flags carry the launch's epoch, so they never need zeroing
    p.sk_epoch = next_sk_epoch();

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    // the kernel waits for the previous one (griddepcontrol.wait) before touching
    // global memory, so its set-up may overlap that kernel's tail
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (kG == 2) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        // run-time tiles: one pair per tile (the running pairs cancel the launches of
        // the rest); otherwise persistent, and with a stream-K tail every co-resident
        // pair takes part
        int grid_clusters = num_tiles;
        if constexpr (!kDyn) {
            const int clusters = concurrent_pairs<kBF16, kIntPath, kRS>(num_sms);
            grid_clusters = (p.sk_tiles > 0 || num_tiles >= clusters) ? clusters : num_tiles;
        }
        cfg.gridDim = dim3(2 * grid_clusters, 1, 1);
    } else {
        const int units = p.sk_tiles > 0 ? num_sms : (num_tiles < num_sms ? num_tiles : num_sms);
        cfg.gridDim = dim3(units, 1, 1);
    }
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int gemm_group_for(int m) { return m > kBM ? 2 : 1; }

int gemm_units(GemmKind kind, int group, int num_sms) {
    if (group == 1) return num_sms;
    switch (kind) {
        case GEMM_F16: return concurrent_pairs<false, false>(num_sms);
        case GEMM_BF16: return concurrent_pairs<true, false>(num_sms);
        case GEMM_RS_F16: return concurrent_pairs<false, false, true>(num_sms);
        case GEMM_RS_BF16: return concurrent_pairs<true, false, true>(num_sms);
        default: return concurrent_pairs<false, true>(num_sms);
    }
}

cudaError_t launch_gemm(GemmKind kind, int group, const GemmParams &p, int num_sms, cudaStream_t stream) {
    if (group == 2) {
        // the plain float GEMM takes its tiles at run time (cluster launch control): on
        // the 28-tile-wide all-gather the slowest persistent pairs had set the time; the
        // reduce-scatter measured no better that way and stays persistent
        switch (kind) {
            case GEMM_F16: return launch_one<2, false, false, false, true>(p, num_sms, stream);
            case GEMM_BF16: return launch_one<2, true, false, false, true>(p, num_sms, stream);
            case GEMM_INT_AS_F16: return launch_one<2, false, true>(p, num_sms, stream);
            case GEMM_RS_F16: return launch_one<2, false, false, true>(p, num_sms, stream);
            case GEMM_RS_BF16: return launch_one<2, true, false, true>(p, num_sms, stream);
        }
    } else {
        switch (kind) {
            case GEMM_F16: return launch_one<1, false, false>(p, num_sms, stream);
            case GEMM_BF16: return launch_one<1, true, false>(p, num_sms, stream);
            case GEMM_INT_AS_F16: return launch_one<1, false, true>(p, num_sms, stream);
            case GEMM_RS_F16: return launch_one<1, false, false, true>(p, num_sms, stream);
            case GEMM_RS_BF16: return launch_one<1, true, false, true>(p, num_sms, stream);
            case GEMM_F16_NARROW: return launch_one<1, false, false, false, false, true>(p, num_sms, stream);
            case GEMM_BF16_NARROW: return launch_one<1, true, false, false, false, true>(p, num_sms, stream);
        }
    }
    return cudaErrorInvalidValue;
}

int *device_status_word() {
    thread_local unsigned long long ready_ctx = 0;
    thread_local int *addr = nullptr;
    const unsigned long long ctx = current_context_id();
    if (ctx == 0 || ctx != ready_ctx) {
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&addr), g_gemm_status) != cudaSuccess) return nullptr;
        ready_ctx = ctx;
    }
    return addr;
}

int read_and_clear_gemm_status(int *status) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_gemm_status, sizeof(int));
    if (e != cudaSuccess) return -1;
    e = cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(int));
    return e == cudaSuccess ? 0 : -1;
}

}  // namespace mc2
