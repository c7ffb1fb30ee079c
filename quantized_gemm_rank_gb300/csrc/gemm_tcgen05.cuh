// gemm_tcgen05.cuh -- the fused MC2 GEMM for sm_103a.
//
// One kernel serves both operations (the tile order is below):
//   * AllGatherMatmul ("torch_npu.npu_all_gather_base_mm", 功能说明/输出说明):
//     A = concat_m of the per-rank chunks, read in place through one TMA
//     tensor map per chunk (or one map, when the chunks lie back to back);
//     out = A @ B (+ bias) rounded to bf16/fp16; the
//     gathered matrix is written from the A tiles already in shared memory
//     (one TMA store per (m-tile, k-tile), by the n-tile-0 tiles only).
//   * AlltoAllQuantMatmul ("aclnnAlltoAllQuantMatmul", 计算公式): A and B
//     hold int8 values as exact fp16; the fp32 tensor-core accumulator stays
//     exact while every partial sum is below 2^24, so the K loop is cut into
//     blocks of at most 1024 (1024 * 127 * 127 < 2^24) and each block's fp32
//     sum is flushed into an int32 register total; the epilogue then applies
//     the per-token x per-channel dequant and the bias in fp32 and rounds to bf16.
//   The float path uses the same K blocks: each block starts from zero in
//   TMEM and the block sums are added in fp32 registers with round-to-nearest,
//   which keeps the tensor core's own accumulation error (it adds at the
//   magnitude of the running sum) to the size of one block's partial sums.
//
// Two shapes of the same kernel (template parameter kG):
//   kG = 1  one CTA per tile: tile 128 x 256 x 64, tcgen05.mma.cta_group::1
//           M=128 N=256, 4-stage ring of 48 KiB stages; or (kNarrow, outputs at
//           most 64 wide) N=64 and an 8-stage ring of 24 KiB stages.
//   kG = 2  a CTA pair (cluster of 2) per tile: tile 256 x 256 x 64,
//           tcgen05.mma.cta_group::2 M=256 N=256 issued by the leader CTA;
//           each CTA loads its own 128 rows of A and 128 rows of B (half the
//           B traffic per CTA of kG = 1), 6-stage ring of 32 KiB stages.
// Tile order (template parameter kDyn):
//   false   persistent: the grid is the co-resident pairs (or CTAs), unit c takes
//           tiles c, c + U, ...; on the integer path the last partial wave is
//           split by K blocks over all units (stream-K, see the Schedule)
//   true    one pair launched per tile; a running pair takes over the tile of a
//           pair that has not launched yet (cluster launch control), so pairs
//           that run faster take more tiles (the plain float GEMM)
// 16-bit operands live in 128-byte-swizzled shared memory; accumulators are
// two 256-column fp32 TMEM buffers per CTA so the epilogue of one K block (or
// tile) overlaps the MMAs of the next.
//
// Warp roles (384 threads per CTA):
//   warp 0      TMA producer (one lane).  Its instruction path per stage bounds
//               the load pipeline, so it issues one copy for A and one for B
//               (N-major B through a 3-D map when n % 64 == 0), with the copy
//               forms fixed at compile time for its k-tile loop.
//   warp 1      TMEM allocator; MMA issuer (the leader CTA for kG = 2): the whole
//               warp runs the issue loop converged and one elected lane issues
//               each tcgen05 instruction (a loop run by a lone lane left the
//               tensor pipe idle ~150 cycles per 512-cycle stage)
//   warp 2      gathered-output TMA store (one lane; AllGather with gather only).
//               On n-tile-0 tiles the MMA commits each stage to a "consumed"
//               barrier instead of "empty"; this warp then stores the A tile
//               (already complete: the MMA read it) and frees the stage, so
//               the store never delays the MMAs.
//   warps 2-3   (weight gradient with its bias gradient) on the first column of
//               tiles, sum each stage's A rows over K from shared memory after
//               the MMAs have read it (the stage comes to them through the same
//               "consumed" barrier), then free it; each tile's sums are the
//               bias gradient of its 128 rows
//   warp 3      otherwise idle
//   warps 4-11  epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (its rows) and
//               half (w-4)/4 of the 256 accumulator columns.  Rounded outputs
//               leave through a swizzled shared slab and a TMA tensor store, but
//               for the reduce-scatter whose warps' rows may span two ranks
//               (stored from registers).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "sm103_ptx.cuh"

namespace mc2 {

constexpr int kBM = 128;  // rows of A per CTA
constexpr int kBN = 256;  // columns of the accumulator (MMA N)
constexpr int kBK = 64;
constexpr int kMaxAMaps = 8;
constexpr int kNumEpiWarps = 8;
constexpr int kNumThreads = 128 + kNumEpiWarps * 32;
constexpr uint32_t kATileBytes = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kTmemCols = 512;              // two 256-column fp32 accumulators
constexpr int kGroupM = 8;                       // m-tiles per raster group (L2 reuse of B) ...
constexpr int kGroupMNarrow = 2;                 // ... and on the float path when the output is at
                                                 // most 16 tiles wide
// Output staging for the TMA-store epilogue: per epilogue warp one 32-row x
// 64-column 16-bit slab (128-byte rows, 128-byte swizzle).
constexpr uint32_t kEpiSlabBytes = 32 * 128;
constexpr uint32_t kEpiStageBytes = kNumEpiWarps * kEpiSlabBytes;

// kTmaOut: reserve the epilogue's shared staging slabs (8 x 4 KiB) after the
// stage ring; every instantiation of the GEMM stores its outputs through them.
// kNarrow (one CTA, outputs at most 64 wide): MMA N = 64 and 24 KiB stages, so
// a ring of 8 holds the whole K of a short problem at once.
template <int kG, bool kTmaOut = false, bool kNarrow = false>
struct TileCfg {
    static constexpr int kTileM = kBM * kG;               // rows per tile
    static constexpr int kMmaN = kNarrow ? 64 : kBN;      // MMA N (accumulator columns written)
    static constexpr int kBRows = kMmaN / kG;             // rows of B (N) per CTA
    static constexpr uint32_t kBTileBytes = kBRows * kBK * 2;
    static constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
    static constexpr int kStages = kNarrow ? 8 : (kG == 1 ? 4 : 6);
    // stages | barriers (1 KiB) | epilogue staging | alignment slack (1 KiB)
    static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024 + (kTmaOut ? kEpiStageBytes : 0) + 1024;
};

// A_SINGLE_MN: one map over an (k, m) row-major matrix, i.e. A = that matrix
// transposed, read M-major (the weight gradient's dY^T)
enum AMode : int { A_SINGLE = 0, A_MCONCAT = 1, A_KINTERLEAVE = 2, A_SINGLE_MN = 3 };

struct GemmParams {
    CUtensorMap a_maps[kMaxAMaps];  // A operand: one map, or one per rank's chunk
    CUtensorMap b_map;              // B operand: (n, k) K-major or (k, n) N-major
    CUtensorMap g_map;              // gathered output (m, k), same box and swizzle as A
    CUtensorMap out_map;            // out (m, n) 16-bit: box 64 columns x 32 rows, 128-byte swizzle
                                    // (every instantiation but the reduce-scatter)
    int num_a_maps;
    int a_mode;
    int a_box_rows;                 // A_MCONCAT: rows per TMA box (divides m_local and kBM)
    int m, n, k;
    int m_local;                    // A_MCONCAT: rows per chunk
    int k_local;                    // A_KINTERLEAVE: columns per chunk
    int b_mn_major;
    int b_3d;                       // N-major B through a 3-D map [n/64][k][64]: one box per stage
    int gather;
    int kblock_tiles;               // integer path: k-tiles per exact fp32 block
    void *out;                      // (m, n): dtype (float path) / bf16 (integer path)
    const void *bias16;             // float path: (n) in the operand dtype, or null
    const float *x1_scale;          // integer path: (m)
    const float *x2_scale;          // integer path: (n)
    const void *bias_q;             // integer path: (n) fp32 or bf16 (required), 16-byte aligned
    int bias_q_bf16;
    int32_t *acc_out;               // integer path: optional (m, n)
    int sk_tiles;                   // integer path: tiles of the stream-K tail (0: whole tiles only)
    int32_t *sk_partials;           // stream-K partial int32 sums: slot (unit * 2 + cta) of 128 x 256,
                                    // lane-contiguous (see the epilogue)
    unsigned long long *sk_flags;   // stream-K, per (tile, cta): (epoch << 24) | parts published; any
                                    // value at launch (a stale epoch counts as none)
    unsigned long long sk_epoch;    // this launch's epoch: unique per launch, in [2^20, 2^40)
    int sk_extra_writers;           // test hook: WRITE parts a FINISH part expects beyond the real ones
                                    // (0 in normal use; > 0 makes every FINISH wait run out)
    int *status;                    // device word set to -7 when a bounded wait gives up
    uint64_t wait_limit_ns;
    // reduce-scatter instantiation only (kRS): B is rank r's weight shard for the
    // k-slice r (same k-interleave as A), and output row i goes to rank
    // i / out_rows at row i % out_rows
    CUtensorMap b_rank_maps[kMaxAMaps];
    void *out_chunks[kMaxAMaps];
    // weight gradient (A = dY^T read M-major): when set, the column sums of dY,
    // i.e. the sums of A's rows over K, rounded once to 16 bits into this (m)
    // vector (the bias gradient)
    void *colsum_out;
    int out_rows;
    // rank r's output (out_rows, n) 16-bit, box 64 columns x 32 rows, 128-byte
    // swizzle; used when rs_tma (out_rows % 32 == 0: a warp's 32 rows are one rank's)
    CUtensorMap out_rank_maps[kMaxAMaps];
    int rs_tma;
};

// ---------------------------------------------------------------------------
// Work schedule of one cluster (identical in every role of every CTA of it).
// Tiles [0, num_tiles - sk_tiles) are data-parallel: cluster c takes tiles
// c, c + U, ... whole.  The K blocks of the last sk_tiles tiles are laid end to
// end and cut into U equal ranges, one per cluster; a range shorter than a
// tile covers at most two parts: the end of one tile and the start of the next.
// A part that does not end at its tile's end is a WRITE part (its int32 sums
// go to the cluster's partial slot); a part that ends there but starts inside
// the tile is a FINISH part (it adds the WRITE parts of the earlier clusters);
// WRITE parts are scheduled first, so a FINISH part never waits on a cluster
// that is itself waiting.
enum WorkKind : int { WORK_FULL = 0, WORK_WRITE = 1, WORK_FINISH = 2 };

struct Work {
    int tile, kb0, kb1, kind;
};

struct Schedule {
    int c, U, nkb, dp_tiles, n_dp, n_sk;
    long long total;  // K blocks in the stream-K region
    Work sk[2];

    __device__ __forceinline__ long long range_start(int u) const { return static_cast<long long>(u) * total / U; }

    __device__ __forceinline__ void init(int cluster, int units, int num_tiles, int sk_tiles, int nkb_) {
        c = cluster;
        U = units;
        nkb = nkb_;
        dp_tiles = num_tiles - sk_tiles;
        n_dp = c < dp_tiles ? (dp_tiles - c + U - 1) / U : 0;
        total = static_cast<long long>(sk_tiles) * nkb;
        n_sk = 0;
        if (sk_tiles == 0) return;
        const long long s0 = range_start(c), e0 = range_start(c + 1);
        if (s0 == e0) return;
        const int t0 = static_cast<int>(s0 / nkb);
        const int kb0 = static_cast<int>(s0 - static_cast<long long>(t0) * nkb);
        const int kb1 = static_cast<int>(min(static_cast<long long>(nkb), kb0 + (e0 - s0)));
        Work a{dp_tiles + t0, kb0, kb1, kb1 < nkb ? WORK_WRITE : (kb0 > 0 ? WORK_FINISH : WORK_FULL)};
        if (e0 > static_cast<long long>(t0 + 1) * nkb) {
            // the range continues into the next tile: that start part is a WRITE part, done first
            Work b{dp_tiles + t0 + 1, 0, static_cast<int>(e0 - static_cast<long long>(t0 + 1) * nkb), WORK_WRITE};
            sk[0] = b;
            sk[1] = a;
            n_sk = 2;
        } else {
            sk[0] = a;
            n_sk = 1;
        }
    }

    __device__ __forceinline__ int count() const { return n_dp + n_sk; }

    __device__ __forceinline__ Work get(int i) const {
        if (i < n_dp) return Work{c + i * U, 0, nkb, WORK_FULL};
        return sk[i - n_dp];
    }

    // Clusters u < c whose non-empty range reaches into `tile` (the WRITE parts a
    // FINISH part of that tile adds), visited in descending u.
    template <class F>
    __device__ __forceinline__ int for_each_writer(int tile, F f) const {
        const long long g0 = static_cast<long long>(tile - dp_tiles) * nkb;
        int n = 0;
        for (int u = c - 1; u >= 0; --u) {
            const long long su = range_start(u), eu = range_start(u + 1);
            if (eu <= g0) break;
            if (su < eu) {
                f(u);
                ++n;
            }
        }
        return n;
    }
};

// Raster order of the tiles: groups of gm m-tiles, each walked m-fastest
// across all n-tiles.  gm is 8 in general.  On the float path with at most 16
// n-tiles (n <= 4096) it is 2, which measured 1-4% faster on each such
// all-gather shape tried (m 8192-16384, k 4096-8192), while on 28-32 n-tiles
// a group of 8 measured 2-5% faster than 2.  The integer path keeps 8 as a
// compile-time constant, which measured 1-2% faster there than either rule.
template <bool kIntPath>
__device__ __forceinline__ int raster_group(int num_n) {
    if constexpr (kIntPath) return kGroupM;
    return num_n <= 16 ? kGroupMNarrow : kGroupM;
}

template <bool kIntPath>
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &mb, int &nb) {
    const int gm = raster_group<kIntPath>(num_n);
    const int span = gm * num_n;
    const int g = tile / span;
    const int first_m = g * gm;
    const int gsz = min(num_m - first_m, gm);
    const int r = tile - g * span;
    mb = first_m + r % gsz;
    nb = r / gsz;
}

// Stream-K publication: one more part of this launch (epoch) written for the
// (tile, cta) flag.  The first publisher of a launch replaces whatever an
// earlier launch left (one compare-and-swap); every later one, and a first
// one that lost that race, adds 1 (only this launch's publishers change the
// flag while it runs, so a failed swap means the flag already holds this
// epoch).  At most two atomics per publisher: a retry loop of swaps among the
// eight epilogue warps of a CTA took several microseconds.
__device__ __forceinline__ void sk_publish(unsigned long long *flag, unsigned long long epoch) {
    const unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(flag);
    if ((cur >> 24) == epoch) {
        atomicAdd(flag, 1ull);
        return;
    }
    if (atomicCAS(flag, cur, (epoch << 24) | 1ull) != cur) atomicAdd(flag, 1ull);
}

// Slow path of a barrier wait: poll with a wall-clock limit and the CTA's
// abort flag; on timeout raise both the flag and the device status word.
template <bool kCluster>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns, int *status,
                                       volatile int *abort_flag) {
    const uint64_t start = ptx::globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - start > limit_ns) {
                *abort_flag = 1;
                if (status) atomicExch(status, -7);
                return false;
            }
        }
    }
}

// Wait for the phase of `bar` with parity `parity`: one try_wait on the fast
// path, the bounded loop otherwise.
template <bool kCluster>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const GemmParams &p,
                                              volatile int *abort_flag) {
    if (kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow<kCluster>(bar, parity, p.wait_limit_ns, p.status, abort_flag);
}

// The work items of one role, in order: the static schedule, or (kDyn) the
// tiles this CTA pair obtains at run time with cluster launch control: its own
// tile first, then each tile whose pair it cancels before that pair launched.
// The leader CTA's producer asks for the next tile when it starts a tile; the
// answer lands in a two-slot ring in both CTAs, and every role of both CTAs
// reads it there when it finishes that tile, then releases the slot on the
// leader's barrier (one release per role).
template <bool kDyn>
struct TileWalk {
    const Schedule *sched;
    int wi;            // static: next schedule index
    int tile;          // dynamic: the current tile, -1 before the first
    int first_tile;    // dynamic: this pair's own tile
    int reads;         // dynamic: answers read so far
    int num_k;
    uint32_t resp0;    // dynamic: the ring's answers (this CTA)
    uint32_t full0;    // dynamic: the ring's arrival barriers (this CTA)
    uint32_t free0;    // dynamic: the ring's release barriers (the leader's, cluster address)
    bool releaser;     // this thread releases the slot for its role

    template <bool kPair>
    __device__ __forceinline__ bool next(Work &w, const GemmParams &p, volatile int *abort_flag) {
        if constexpr (!kDyn) {
            if (wi >= sched->count()) return false;
            w = sched->get(wi++);
            return true;
        } else {
            if (tile < 0) {
                tile = first_tile;
                w = Work{tile, 0, (num_k + p.kblock_tiles - 1) / p.kblock_tiles, WORK_FULL};
                return true;
            }
            const int j = reads & 1;
            const unsigned mask = __activemask();
            const bool got = __all_sync(mask, wait_or_abort<false>(full0 + 8u * j, (reads >> 1) & 1, p, abort_flag));
            uint32_t x = 0;
            const bool more = got && ptx::clc_query(resp0 + 16u * j, x);
            __syncwarp(mask);
            if (releaser && got) ptx::mbar_arrive_remote_relaxed(free0 + 8u * j);
            ++reads;
            if (!more) return false;
            tile = static_cast<int>(x) / (kPair ? 2 : 1);
            w = Work{tile, 0, (num_k + p.kblock_tiles - 1) / p.kblock_tiles, WORK_FULL};
            return true;
        }
    }
};

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (kBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    } else {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
}

template <bool kBF16>
__device__ __forceinline__ float load16(const void *base, int idx) {
    const uint16_t v = reinterpret_cast<const uint16_t *>(base)[idx];
    if constexpr (kBF16) {
        return __uint_as_float(static_cast<uint32_t>(v) << 16);
    } else {
        return __half2float(__ushort_as_half(v));
    }
}

// Store 32 consecutive 16-bit outputs (columns col0 .. col0+31) of the row that
// starts at row_ptr, masked at n.
__device__ __forceinline__ void store_row32_16(uint16_t *row_ptr, int n, int col0, const uint32_t (&pk)[16]) {
    uint16_t *dst = row_ptr + col0;
    if (col0 + 32 <= n) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int j = 0; j < 4; ++j) d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < n) dst[i] = static_cast<uint16_t>((pk[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu);
    }
}

// kDyn: one CTA pair launched per tile, balanced at run time by cluster launch
// control (float path only: no stream-K tail).  kNarrow: see TileCfg (float
// path, one CTA per tile, n <= 64).
template <int kG, bool kBF16, bool kIntPath, bool kRS = false, bool kDyn = false, bool kNarrow = false>
__global__ void __launch_bounds__(kNumThreads, 1) mc2_gemm_kernel(const __grid_constant__ GemmParams p) {
    static_assert(!kDyn || (kG == 2 && !kIntPath), "run-time tiles are a CTA-pair float-path form");
    static_assert(!kNarrow || (kG == 1 && !kIntPath && !kRS && !kDyn), "the narrow tile is a one-CTA float-path form");
    constexpr bool kTmaOut = true;  // epilogue stores through shared slabs and TMA (see the epilogue)
    using Cfg = TileCfg<kG, kTmaOut, kNarrow>;
    constexpr bool kPair = kG == 2;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * Cfg::kStageBytes);
    uint64_t *full_bar = bars;                // A/B of the stage landed (the leader's counts both CTAs)
    uint64_t *empty_bar = bars + S;           // stage free in this CTA
    uint64_t *consumed_bar = bars + 2 * S;    // gathered tiles: the MMAs have read the stage
    uint64_t *tfull_bar = bars + 3 * S;       // accumulator buffer ready
    uint64_t *tempty_bar = bars + 3 * S + 2;  // accumulator buffer drained (the leader's counts both CTAs)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * S + 4);
    uint64_t *drain_bar = bars + 3 * S + 5;   // every MMA this CTA issued has completed
    uint64_t *skr_bar = bars + 3 * S + 6;     // per epilogue warp: its share of a stream-K partial landed
    uint64_t *walk_resp = bars + 3 * S + 14;  // kDyn: two 16-byte answers (16-byte aligned)
    uint64_t *walk_full = bars + 3 * S + 18;  // kDyn: answer landed (this CTA)
    uint64_t *walk_free = bars + 3 * S + 20;  // kDyn: answer read by every role (the leader's counts both CTAs)
    // the epilogue's output slabs, after the 1 KiB barrier area (1024-byte aligned)
    uint8_t *epi_stage = smem + S * Cfg::kStageBytes + 1024;
    __shared__ int abort_flag_s;
    volatile int *abort_flag = &abort_flag_s;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t cr = kPair ? ptx::cluster_ctarank() : 0u;  // rank inside the pair
    const bool leader = cr == 0;
    const int num_m = (p.m + Cfg::kTileM - 1) / Cfg::kTileM;
    const int num_n = (p.n + kBN - 1) / kBN;
    const int num_tiles = num_m * num_n;
    const int num_k = (p.k + kBK - 1) / kBK;
    const int cluster_id = blockIdx.x / kG;
    const int num_clusters = gridDim.x / kG;
    const int nkb = (num_k + p.kblock_tiles - 1) / p.kblock_tiles;  // K blocks per tile
    Schedule sched;
    sched.init(cluster_id, num_clusters, num_tiles, p.sk_tiles, nkb);
    // every role walks its own copy
    TileWalk<kDyn> walk0;
    walk0.sched = &sched;
    walk0.wi = 0;
    walk0.tile = -1;
    walk0.first_tile = cluster_id;
    walk0.reads = 0;
    walk0.num_k = num_k;
    walk0.resp0 = ptx::smem_u32(&walk_resp[0]);
    walk0.full0 = ptx::smem_u32(&walk_full[0]);
    walk0.free0 = kPair ? ptx::mapa(ptx::smem_u32(&walk_free[0]), 0) : ptx::smem_u32(&walk_free[0]);
    walk0.releaser = lane == 0;

    if (threadIdx.x == 0) {
        abort_flag_s = 0;
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&consumed_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&tfull_bar[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&tempty_bar[b]), kNumEpiWarps * kG);
        }
        ptx::mbar_init(ptx::smem_u32(drain_bar), 1);
        for (int e = 0; e < kNumEpiWarps; ++e) ptx::mbar_init(ptx::smem_u32(&skr_bar[e]), 1);
        if constexpr (kDyn) {
            // releases per answer: per CTA the producer, the epilogue warps and the
            // gathered-store lane, plus the leader's MMA warp
            const uint32_t roles = kG * (1 + kNumEpiWarps + (p.gather ? 1 : (p.colsum_out ? 2 : 0))) + 1;
            for (int j = 0; j < 2; ++j) {
                ptx::mbar_init(ptx::smem_u32(&walk_full[j]), 1);
                ptx::mbar_init(ptx::smem_u32(&walk_free[j]), roles);
            }
        }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc<kG>(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish<kG>();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (kPair) ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // The set-up above may overlap the previous kernel of the stream; nothing in
    // global memory is touched before it has completed.
    ptx::grid_dependency_wait();
    // The next kernel of the stream may be scheduled from now on: its CTAs take
    // the SMs this grid leaves, and it waits for this grid to complete before
    // it touches global memory.
    ptx::allow_dependent_launch();

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        for (int i = 0; i < p.num_a_maps; ++i) ptx::prefetch_tmap(&p.a_maps[i]);
        if constexpr (kRS) {
            for (int i = 0; i < p.num_a_maps; ++i) ptx::prefetch_tmap(&p.b_rank_maps[i]);
        } else {
            ptx::prefetch_tmap(&p.b_map);
        }
        // bytes that complete the leader's full barrier per stage (both CTAs' tiles)
        constexpr uint32_t leader_bytes = Cfg::kStageBytes * kG;
        int stage = 0;
        uint32_t phase = 0;
        int iters = 0;
        bool ok = true;
        // B copy form, fixed for the launch: 0 K-major box, 1 N-major boxes, 2 one 3-D N-major box
        const int b_mode = !p.b_mn_major ? 0 : (p.b_3d ? 2 : 1);
        // A form: the AMode, with the all-gather split into one box per k-tile (4) or several
        const int a_form = p.a_mode == A_MCONCAT && p.a_box_rows == kBM ? 4 : p.a_mode;
        // addresses of stage 0 (stage s adds s * 8 to a barrier, s * kStageBytes to a tile);
        // the pair's peer signals the leader's full barrier at the same offset
        const uint32_t full0 = ptx::smem_u32(&full_bar[0]);
        const uint32_t empty0 = ptx::smem_u32(&empty_bar[0]);
        const uint32_t sA0 = ptx::smem_u32(smem);
        const uint32_t sig0 = (kPair && !leader) ? ptx::mapa(full0, 0) : full0;
        auto load = [&](uint32_t dst, const CUtensorMap *m, int c0, int c1, uint32_t bar) {
            if constexpr (kPair)
                ptx::tma_load_2d_pair(dst, m, c0, c1, bar);
            else
                ptx::tma_load_2d(dst, m, c0, c1, bar);
        };
        // one work tile's k-tiles, with the copy forms as compile-time constants
        auto k_loop = [&](auto a_c, auto b_c, int kt_begin, int kt_end, int m0, int n0, int a_chunk0, int a_row0,
                          int a_nbox, int kc, int kl) {
            constexpr int AF = decltype(a_c)::value;
            constexpr int BF = decltype(b_c)::value;
            for (int kt = kt_begin; kt < kt_end; ++kt) {
                // (CTA scope: the stage is released by the MMA's tcgen05.commit)
                if (!wait_or_abort<false>(empty0 + 8u * stage, phase ^ 1u, p, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sA = sA0 + stage * Cfg::kStageBytes;
                const uint32_t sB = sA + kATileBytes;
                const uint32_t bar = sig0 + 8u * stage;
                if (leader) ptx::mbar_arrive_expect_tx(full0 + 8u * stage, leader_bytes);
                const int k0 = kt * kBK;
                if constexpr (AF == 4) {
                    load(sA, &p.a_maps[a_chunk0], k0, a_row0, bar);
                } else if constexpr (AF == A_MCONCAT) {
                    // walk the tile's boxes through the chunks (box_rows divides m_local)
                    int c = a_chunk0, li = a_row0;
                    for (int j = 0; j < a_nbox; ++j) {
                        load(sA + j * p.a_box_rows * 128, &p.a_maps[c], k0, li, bar);
                        li += p.a_box_rows;
                        if (li >= p.m_local && c < p.num_a_maps - 1) li -= p.m_local, ++c;
                    }
                } else if constexpr (AF == A_KINTERLEAVE) {
                    // permuted column k0 = kc * k_local + kl lives in chunk kc (k_local % kBK == 0)
                    load(sA, &p.a_maps[kc], kl, m0, bar);
                    if constexpr (kRS) {
                        // ... and so does the B slice: rank kc's weight shard at column kl
                        const CUtensorMap *bm = &p.b_rank_maps[kc];
                        if constexpr (BF != 0) {
#pragma unroll
                            for (int j = 0; j < Cfg::kBRows / 64; ++j)
                                load(sB + j * (kBK * 128), bm, n0 + 64 * j, kl, bar);
                        } else {
                            load(sB, bm, kl, n0, bar);
                        }
                    }
                    kl += kBK;
                    if (kl >= p.k_local) kl = 0, ++kc;
                } else if constexpr (AF == A_SINGLE_MN) {
                    // M-major A: 64-wide M slabs of the (k, m) matrix, like an N-major B
#pragma unroll
                    for (int j = 0; j < kBM / 64; ++j) load(sA + j * (kBK * 128), &p.a_maps[0], m0 + 64 * j, k0, bar);
                } else {
                    load(sA, &p.a_maps[0], k0, m0, bar);
                }
                if constexpr (!kRS) {
                    if constexpr (BF == 0) {
                        load(sB, &p.b_map, k0, n0, bar);
                    } else if constexpr (BF == 2) {
                        // all kBRows / 64 column groups in one copy, group j at sB + j * 8 KiB
                        if constexpr (kPair)
                            ptx::tma_load_3d_pair(sB, &p.b_map, 0, k0, n0 >> 6, bar);
                        else
                            ptx::tma_load_3d(sB, &p.b_map, 0, k0, n0 >> 6, bar);
                    } else {
#pragma unroll
                        for (int j = 0; j < Cfg::kBRows / 64; ++j)
                            load(sB + j * (kBK * 128), &p.b_map, n0 + 64 * j, k0, bar);
                    }
                }
                ++iters;
                if (++stage == S) stage = 0, phase ^= 1u;
            }
        };
        TileWalk<kDyn> walk = walk0;
        int asked = 0;   // kDyn: answers asked for (one per tile started)
        Work w;
        while (ok && walk.template next<kPair>(w, p, abort_flag)) {
            if constexpr (kDyn) {
                // ask for the tile after this one: the answer goes to slot asked & 1 of both CTAs
                const uint32_t j = asked & 1;
                const uint32_t wf = ptx::smem_u32(&walk_full[j]);
                if (leader) {
                    if (!wait_or_abort<false>(ptx::smem_u32(&walk_free[j]), ((asked >> 1) & 1) ^ 1u, p, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(wf, 16);
                    ptx::clc_try_cancel_multicast(ptx::smem_u32(&walk_resp[2 * j]), wf);
                } else {
                    ptx::mbar_arrive_expect_tx(wf, 16);
                }
                ++asked;
            }
            const int kt_begin = w.kb0 * p.kblock_tiles, kt_end = min(num_k, w.kb1 * p.kblock_tiles);
            int mb, nb;
            tile_coords<kIntPath>(w.tile, num_m, num_n, mb, nb);
            const int m0 = mb * Cfg::kTileM + kBM * static_cast<int>(cr);
            const int n0 = nb * kBN + Cfg::kBRows * static_cast<int>(cr);
            // first A box of this tile: chunk and row inside it (rows past m stay in the
            // last chunk, out of its range, and read as zeros)
            int a_chunk0 = 0, a_row0 = m0, a_nbox = 1;
            int kc = 0, kl = 0;  // A_KINTERLEAVE: chunk and column inside it of the current k-tile
            if (p.a_mode == A_KINTERLEAVE) {
                kc = kt_begin * kBK / p.k_local;
                kl = kt_begin * kBK - kc * p.k_local;
            }
            if (p.a_mode == A_MCONCAT) {
                a_chunk0 = m0 / p.m_local;
                a_row0 = m0 - a_chunk0 * p.m_local;
                if (a_chunk0 > p.num_a_maps - 1) {
                    a_row0 += (a_chunk0 - (p.num_a_maps - 1)) * p.m_local;
                    a_chunk0 = p.num_a_maps - 1;
                }
                a_nbox = kBM / p.a_box_rows;
            }
            using I0 = std::integral_constant<int, 0>;
            using I1 = std::integral_constant<int, 1>;
            using I2 = std::integral_constant<int, 2>;
            auto with_b = [&](auto a_c) {
                if (b_mode == 0)
                    k_loop(a_c, I0{}, kt_begin, kt_end, m0, n0, a_chunk0, a_row0, a_nbox, kc, kl);
                else if (b_mode == 2)
                    k_loop(a_c, I2{}, kt_begin, kt_end, m0, n0, a_chunk0, a_row0, a_nbox, kc, kl);
                else
                    k_loop(a_c, I1{}, kt_begin, kt_end, m0, n0, a_chunk0, a_row0, a_nbox, kc, kl);
            };
            switch (a_form) {
                case 4: with_b(std::integral_constant<int, 4>{}); break;
                case A_MCONCAT: with_b(std::integral_constant<int, A_MCONCAT>{}); break;
                case A_KINTERLEAVE: with_b(std::integral_constant<int, A_KINTERLEAVE>{}); break;
                case A_SINGLE_MN: with_b(std::integral_constant<int, A_SINGLE_MN>{}); break;
                default: with_b(std::integral_constant<int, A_SINGLE>{}); break;
            }
        }
        if (!ok) {
            // let the copies already in flight land before the CTA can exit
            const bool armed_local = leader;
            for (int back = 1; back <= S && back <= iters && armed_local; ++back) {
                const int i = iters - back;
                (void)ptx::mbar_wait(ptx::smem_u32(&full_bar[i % S]), static_cast<uint32_t>((i / S) & 1),
                                     p.wait_limit_ns);
            }
            ptx::nanosleep(20000);
        }
    } else if (warp == 1 && leader) {
        // ------------------------------------------------------------ MMA issuer
        const bool a_mn = p.a_mode == A_SINGLE_MN;
        const uint32_t idesc = ptx::idesc_f16(kBF16 && !kIntPath, p.b_mn_major != 0, Cfg::kTileM, Cfg::kMmaN, a_mn);
        // descriptors of stage 0, k-slice 0; later ones add to the address field
        // (>> 4 units): per 16-wide k-slice +2 (K-major: 32 bytes into the
        // swizzled row) or +128 (MN-major: 16 rows of 128 bytes), +stage bytes per stage
        const uint32_t s0 = ptx::smem_u32(smem);
        const uint64_t a_desc0 = a_mn ? ptx::smem_desc_sw128(s0, kBK * 128, 1024) : ptx::smem_desc_sw128(s0, 16, 1024);
        const uint32_t a_kk = a_mn ? (2048u >> 4) : (32u >> 4);
        const uint64_t b_desc0 = p.b_mn_major ? ptx::smem_desc_sw128(s0 + kATileBytes, kBK * 128, 1024)
                                              : ptx::smem_desc_sw128(s0 + kATileBytes, 16, 1024);
        const uint32_t b_kk = p.b_mn_major ? (2048u >> 4) : (32u >> 4);
        constexpr uint32_t kStageStep = Cfg::kStageBytes >> 4;
        const uint32_t full0 = ptx::smem_u32(&full_bar[0]);
        const uint32_t empty0 = ptx::smem_u32(&empty_bar[0]);
        const int kblock = p.kblock_tiles;
        int stage = 0;
        uint32_t phase = 0, stage_off = 0;
        uint32_t acc_iter = 0;
        bool ok = true;
        uint32_t d_tmem = tmem_base;
        const uint32_t consumed0 = ptx::smem_u32(&consumed_bar[0]);
        TileWalk<kDyn> walk = walk0;
        Work w;
        while (ok && walk.template next<kPair>(w, p, abort_flag)) {
            const int kt_begin = w.kb0 * kblock, kt_end = min(num_k, w.kb1 * kblock);
            int mb, nb;
            tile_coords<kIntPath>(w.tile, num_m, num_n, mb, nb);
            // stages of gathered tiles go to the gathered-store warp, and those of bias-gradient
            // tiles to the summing warps, before being freed
            const uint32_t release0 = ((p.gather || p.colsum_out != nullptr) && nb == 0) ? consumed0 : empty0;
            int kin = 0;  // k-tile index inside the current K block
            for (int kt = kt_begin; kt < kt_end; ++kt) {
                if (kin == 0) {
                    const uint32_t b = acc_iter & 1u;
                    const bool got = wait_or_abort<kPair>(ptx::smem_u32(&tempty_bar[b]), ((acc_iter >> 1) & 1u) ^ 1u,
                                                          p, abort_flag);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    d_tmem = tmem_base + b * kBN;
                }
                // (CTA scope: the stage is completed by the copies' transaction bytes)
                const bool gotf = wait_or_abort<false>(full0 + 8u * stage, phase, p, abort_flag);
                if (!__all_sync(0xffffffffu, gotf)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t ad = a_desc0 + stage_off;
                const uint64_t bd = b_desc0 + stage_off;
                ptx::mma_f16_ss<kG>(d_tmem, ad, bd, idesc, kin > 0 ? 1u : 0u);
                ptx::mma_f16_ss<kG>(d_tmem, ad + a_kk, bd + b_kk, idesc, 1u);
                ptx::mma_f16_ss<kG>(d_tmem, ad + 2 * a_kk, bd + 2 * b_kk, idesc, 1u);
                ptx::mma_f16_ss<kG>(d_tmem, ad + 3 * a_kk, bd + 3 * b_kk, idesc, 1u);
                ptx::mma_commit<kG>(release0 + 8u * stage);
                if (++stage == S) {
                    stage = 0;
                    stage_off = 0;
                    phase ^= 1u;
                } else {
                    stage_off += kStageStep;
                }
                if (++kin == kblock || kt == kt_end - 1) {
                    ptx::mma_commit<kG>(ptx::smem_u32(&tfull_bar[acc_iter & 1u]));
                    ++acc_iter;
                    kin = 0;
                }
            }
        }
        // Drain: whether the loop ended or gave up, wait (bounded) until every MMA
        // issued above has completed, so that no MMA can still write TMEM (in
        // either CTA of a pair) when the CTAs pass the final barrier and free it.
        // On the normal path they have all completed already (the epilogue waited
        // for their accumulators) and this returns at once.
        ptx::mma_commit_local<kG>(ptx::smem_u32(drain_bar));
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(drain_bar), 0u, p.wait_limit_ns))) {
            *abort_flag = 1;
            if (p.status && lane == 0) atomicExch(p.status, -7);
        }
    } else if ((warp == 2 || warp == 3) && p.colsum_out != nullptr) {
        // ------------------------------------------------------------ bias gradient
        // A is dY^T read M-major: a stage holds, per CTA, two 64-column slabs of dY
        // (its 128 output rows), 64 dY rows of 128 bytes each, 128-byte swizzled (chunk
        // c of row r at chunk c ^ (r % 8)).  Warp 2 sums slab 0 and warp 3 slab 1: lane
        // (c = l % 8, g = l / 8) adds chunk c of rows g, g + 4, ... (16 per stage) into
        // 8 fp32 sums; at the tile's end the 4 row groups are added (lanes g = 0..3)
        // and rounded once.  Fixed order: the result is deterministic.
        const int slab = warp - 2;
        const int c = lane & 7;
        const int g = lane >> 3;
        int stage = 0;
        uint32_t consumed_parity = 0;  // bit s: parity of the next consumed_bar[s] phase
        bool ok = true;
        TileWalk<kDyn> walk = walk0;
        Work w;
        while (ok) {
            // the two warps take each tile together: with tiles obtained at run time
            // one of them could see an abort that the other does not, and would
            // leave the other waiting alone at the named barrier below
            if (!ptx::bar_red_and(1, 64, walk.template next<kPair>(w, p, abort_flag))) break;
            const int kt_begin = w.kb0 * p.kblock_tiles, kt_end = min(num_k, w.kb1 * p.kblock_tiles);
            int mb, nb;
            tile_coords<kIntPath>(w.tile, num_m, num_n, mb, nb);
            if (nb != 0) {  // its stages are freed by the MMA directly
                stage = (stage + (kt_end - kt_begin)) % S;
                continue;
            }
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
            for (int kt = kt_begin; kt < kt_end; ++kt) {
                const bool got = __all_sync(0xffffffffu, wait_or_abort<kPair>(ptx::smem_u32(&consumed_bar[stage]),
                                                                              (consumed_parity >> stage) & 1u, p,
                                                                              abort_flag));
                if (got) {
                    const uint8_t *slab_p = smem + stage * Cfg::kStageBytes + slab * (kBK * 128);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int r = g + 4 * i;
                        const uint4 v = *reinterpret_cast<const uint4 *>(slab_p + r * 128 + ((c ^ (r & 7)) << 4));
                        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float lo, hi;
                            if constexpr (kBF16) {
                                lo = __uint_as_float(vw[e] << 16);
                                hi = __uint_as_float(vw[e] & 0xFFFF0000u);
                            } else {
                                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&vw[e]));
                                lo = f.x;
                                hi = f.y;
                            }
                            acc[2 * e] = __fadd_rn(acc[2 * e], lo);
                            acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], hi);
                        }
                    }
                }
                // both warps have read the stage (or both give up): the stage is free
                if (!ptx::bar_red_and(1, 64, got)) {
                    ok = false;
                    break;
                }
                consumed_parity ^= 1u << stage;
                if (warp == 2 && lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty_bar[stage]));
                if (++stage == S) stage = 0;
            }
            if (!ok) break;
            // the four row groups of each chunk, in a fixed order
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                acc[e] = __fadd_rn(acc[e], __shfl_xor_sync(0xffffffffu, acc[e], 8));
                acc[e] = __fadd_rn(acc[e], __shfl_xor_sync(0xffffffffu, acc[e], 16));
            }
            const int col = mb * Cfg::kTileM + kBM * static_cast<int>(cr) + 64 * slab + 8 * c;
            if (g == 0 && col < p.m) {
                uint4 o;
                o.x = pack2<kBF16>(acc[0], acc[1]);
                o.y = pack2<kBF16>(acc[2], acc[3]);
                o.z = pack2<kBF16>(acc[4], acc[5]);
                o.w = pack2<kBF16>(acc[6], acc[7]);
                *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.colsum_out) + col) = o;
            }
        }
    } else if (warp == 2 && lane == 0 && p.gather) {
        // ------------------------------------------------------------ gathered store
        ptx::prefetch_tmap(&p.g_map);
        int stage = 0;
        uint32_t consumed_parity = 0;  // bit s: parity of the next consumed_bar[s] phase
        int pending_stage = -1;        // stage whose store may still be reading shared memory
        bool ok = true;
        TileWalk<kDyn> walk = walk0;
        Work w;
        while (ok && walk.template next<kPair>(w, p, abort_flag)) {
            const int kt_begin = w.kb0 * p.kblock_tiles, kt_end = min(num_k, w.kb1 * p.kblock_tiles);
            int mb, nb;
            tile_coords<kIntPath>(w.tile, num_m, num_n, mb, nb);
            if (nb != 0) {  // not a gathered tile: its stages are freed by the MMA directly
                stage = (stage + (kt_end - kt_begin)) % S;
                continue;
            }
            const int m0 = mb * Cfg::kTileM + kBM * static_cast<int>(cr);
            for (int kt = kt_begin; kt < kt_end; ++kt) {
                if (!wait_or_abort<kPair>(ptx::smem_u32(&consumed_bar[stage]), (consumed_parity >> stage) & 1u, p,
                                          abort_flag)) {
                    ok = false;
                    break;
                }
                consumed_parity ^= 1u << stage;
                ptx::tma_store_2d(&p.g_map, kt * kBK, m0, ptx::smem_u32(smem + stage * Cfg::kStageBytes));
                ptx::bulk_commit_group();
                // free the previous stage once its store has finished reading it
                ptx::bulk_wait_group_read<1>();
                if (pending_stage >= 0) ptx::mbar_arrive(ptx::smem_u32(&empty_bar[pending_stage]));
                pending_stage = stage;
                if (++stage == S) stage = 0;
            }
            ptx::bulk_wait_group_read<0>();
            if (pending_stage >= 0) ptx::mbar_arrive(ptx::smem_u32(&empty_bar[pending_stage]));
            pending_stage = -1;
        }
        ptx::bulk_wait_group<0>();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quadrant this warp may access
        const int half = (warp - 4) >> 2;     // which 128 of the 256 columns
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        uint32_t acc_iter = 0;
        uint32_t skr_phase = 0;   // phase of this warp's stream-K partial barrier
        TileWalk<kDyn> walk = walk0;
        Work w;
        while (walk.template next<kPair>(w, p, abort_flag)) {
            int mb, nb;
            tile_coords<kIntPath>(w.tile, num_m, num_n, mb, nb);
            const int row = mb * Cfg::kTileM + kBM * static_cast<int>(cr) + 32 * q + lane;
            const int colh = nb * kBN + half * 128;
            bool ok = true;
            if constexpr (kIntPath) {
                // This warp's 128 column scales and biases are read only after the tile's
                // last K block; fetching their lines into L1 now takes those reads (eight
                // dependent ones per thread) off the tile's critical path.
                if (lane < 8 && w.kind != WORK_WRITE) {
                    const int c = min(colh + 16 * lane, p.n - 1);
                    ptx::prefetch_l1(p.x2_scale + c);
                    ptx::prefetch_l1(p.bias_q_bf16 ? static_cast<const void *>(static_cast<const uint16_t *>(p.bias_q) + c)
                                                   : static_cast<const void *>(static_cast<const float *>(p.bias_q) + c));
                }
            }
            // Sum of the K blocks: exact int32 (integer path) or fp32 with
            // round-to-nearest adds (float path); one TMEM drain per block.
            using acc_t = typename std::conditional<kIntPath, int32_t, float>::type;
            acc_t sum[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) sum[i] = acc_t(0);
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                const uint32_t b = acc_iter & 1u;
                // every lane waits (bounded); the warp goes on only if all of them saw the
                // buffer ready, so no lane reaches the warp-wide TMEM load alone
                const bool got = wait_or_abort<kPair>(ptx::smem_u32(&tfull_bar[b]), (acc_iter >> 1) & 1u, p, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // 16 columns per TMEM load: with the 128 running sums live, a 32-column
                // load pushed the epilogue past its registers into local memory
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if (colh + c * 16 < p.n) {
                        uint32_t r[16];
                        ptx::tmem_ld_32x32b_x16(tmem_base + lane_addr + b * kBN + half * 128 + c * 16, r);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if constexpr (kIntPath)
                                sum[c * 16 + i] += __float2int_rn(__uint_as_float(r[i]));
                            else
                                sum[c * 16 + i] = __fadd_rn(sum[c * 16 + i], __uint_as_float(r[i]));
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)
                        ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_u32(&tempty_bar[b]), 0));
                    else
                        ptx::mbar_arrive(ptx::smem_u32(&tempty_bar[b]));
                }
                ++acc_iter;
            }
            if (!ok) break;
            if constexpr (kIntPath) {
                if (w.kind != WORK_FULL) {
                    // stream-K: this thread's 128 int32 sums in slot (unit, cta), laid out
                    // lane-contiguous (vector j of epilogue warp e, lane l at int4 index
                    // (e * 32 + j) * 32 + l), so a warp's store or load is 512 contiguous bytes
                    const size_t lane_off = static_cast<size_t>(warp - 4) * 32 * 32 + lane;
                    if (w.kind == WORK_WRITE) {
                        int4 *slot = reinterpret_cast<int4 *>(p.sk_partials +
                                                              static_cast<size_t>(cluster_id * 2 + cr) * kBM * kBN) +
                                     lane_off;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            __stcg(slot + j * 32, make_int4(sum[4 * j], sum[4 * j + 1], sum[4 * j + 2], sum[4 * j + 3]));
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) sk_publish(p.sk_flags + w.tile * 2 + cr, p.sk_epoch);
                        continue;
                    }
                    // FINISH: wait until every epilogue warp of every earlier part has published.
                    // Lane 0 polls (bounded) and tells the warp, so the warp decides as one.
                    const int writers = sched.for_each_writer(w.tile, [](int) {}) + p.sk_extra_writers;
                    const unsigned long long want =
                        (p.sk_epoch << 24) | static_cast<unsigned long long>(kNumEpiWarps * writers);
                    int seen = 1;
                    if (lane == 0) {
                        volatile unsigned long long *flag = p.sk_flags + w.tile * 2 + cr;
                        if (*flag != want) {
                            const uint64_t start = ptx::globaltimer_ns();
                            while (*flag != want) {
                                if (*abort_flag || ptx::globaltimer_ns() - start > p.wait_limit_ns) {
                                    *abort_flag = 1;
                                    if (p.status) atomicExch(p.status, -7);
                                    seen = 0;
                                    break;
                                }
                                ptx::nanosleep(64);
                            }
                        }
                    }
                    if (__shfl_sync(0xffffffffu, seen, 0) == 0) {
                        ok = false;
                        break;
                    }
                    // The earlier parts' sums (exact int32: the order does not matter).  This is
                    // the unit's last work item and its own MMAs have completed, so the stage
                    // ring is idle: each writer's share for this warp (16 KiB, contiguous in its
                    // slot) comes in with one bulk copy into this warp's 16 KiB of the ring, and
                    // is added from shared memory (one round trip instead of a chain of them).
                    const uint32_t area = ptx::smem_u32(smem) + static_cast<uint32_t>(warp - 4) * 16384u;
                    const uint32_t wbar = ptx::smem_u32(&skr_bar[warp - 4]);
                    if (lane == 0) {
                        __threadfence();                   // acquire: the writers' data, seen through the flag ...
                        ptx::fence_proxy_async_global();   // ... before the bulk copies read it
                    }
                    bool got_all = true;
                    sched.for_each_writer(w.tile, [&](int u) {
                        if (!got_all) return;
                        if (lane == 0) {
                            ptx::mbar_arrive_expect_tx(wbar, 16384u);
                            ptx::bulk_load_1d(area,
                                              reinterpret_cast<const int4 *>(p.sk_partials +
                                                                             static_cast<size_t>(u * 2 + cr) * kBM * kBN) +
                                                  static_cast<size_t>(warp - 4) * 32 * 32,
                                              16384u, wbar);
                        }
                        if (!__all_sync(0xffffffffu, ptx::mbar_wait(wbar, skr_phase, p.wait_limit_ns))) {
                            got_all = false;
                            return;
                        }
                        skr_phase ^= 1u;
                        const int4 *sv = reinterpret_cast<const int4 *>(smem + static_cast<size_t>(warp - 4) * 16384u);
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int4 v = sv[j * 32 + lane];
                            sum[4 * j] += v.x;
                            sum[4 * j + 1] += v.y;
                            sum[4 * j + 2] += v.z;
                            sum[4 * j + 3] += v.w;
                        }
                        // the area is read before the next copy overwrites it
                        __syncwarp();
                        ptx::fence_proxy_async_smem();
                    });
                    if (!got_all) {
                        *abort_flag = 1;
                        if (p.status && lane == 0) atomicExch(p.status, -7);
                        ptx::nanosleep(20000);   // a copy still in flight lands before the CTA exits
                        ok = false;
                        break;
                    }
                }
            }
            const bool row_ok = row < p.m;
            // the reduce-scatter with out_rows % 32 != 0 writes rows straight from
            // registers (a warp's rows may belong to two ranks)
            const bool rs_direct = kRS && !p.rs_tma;
            if (rs_direct && !row_ok) continue;   // no warp-wide steps below in that mode
            // This warp's 32 rows x 128 columns leave as two 64-column slabs:
            // rounded 16-bit values go to its shared staging slab (128-byte rows,
            // chunk j of row r at ((j ^ (r % 8)) * 16)), then one TMA store per
            // slab; rows and columns past the output are clipped by the TMA unit.
            // The reduce-scatter stores through the map of the rank that owns the
            // warp's rows, at the rows' place in that rank's output.
            uint8_t *slab = reinterpret_cast<uint8_t *>(epi_stage) + (warp - 4) * kEpiSlabBytes;
            const int slab_row0 = mb * Cfg::kTileM + kBM * static_cast<int>(cr) + 32 * q;
            const CUtensorMap *omap = &p.out_map;
            int orow0 = slab_row0;
            bool ostore = true;
            if constexpr (kRS) {
                const int rank = min(slab_row0 / p.out_rows, p.num_a_maps - 1);
                omap = &p.out_rank_maps[rank];
                orow0 = slab_row0 - rank * p.out_rows;
                ostore = slab_row0 < p.m;   // warp-uniform: out_rows % 32 == 0 in this mode
            }
            auto put = [&](int c, const uint32_t (&pk)[16]) {
                if (rs_direct) {
                    uint16_t *orow = reinterpret_cast<uint16_t *>(p.out_chunks[row / p.out_rows]) +
                                     static_cast<int64_t>(row % p.out_rows) * p.n;
                    store_row32_16(orow, p.n, colh + c * 32, pk);
                } else {
                    if ((c & 1) == 0) {
                        // the slab's previous store has finished reading it
                        if (lane == 0) ptx::bulk_wait_group_read<0>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int j16 = (c & 1) * 4 + j;
                        *reinterpret_cast<uint4 *>(slab + lane * 128 + ((j16 ^ (lane & 7)) << 4)) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                    if ((c & 1) == 1) {
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        const int scol = colh + (c >> 1) * 64;
                        if (lane == 0 && ostore && scol < p.n) {
                            ptx::tma_store_2d(omap, scol, orow0, ptx::smem_u32(slab));
                            ptx::bulk_commit_group();
                        }
                    }
                }
            };
            if constexpr (!kIntPath) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int col0 = colh + c * 32;
                    if (rs_direct && col0 >= p.n) continue;
                    uint32_t pk[16];
                    if (p.bias16 != nullptr) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack2<kBF16>(
                                __fadd_rn(sum[c * 32 + 2 * i], load16<kBF16>(p.bias16, min(col0 + 2 * i, p.n - 1))),
                                __fadd_rn(sum[c * 32 + 2 * i + 1],
                                          load16<kBF16>(p.bias16, min(col0 + 2 * i + 1, p.n - 1))));
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[i] = pack2<kBF16>(sum[c * 32 + 2 * i], sum[c * 32 + 2 * i + 1]);
                    }
                    put(c, pk);
                }
            } else {
                const float s1 = row_ok ? p.x1_scale[row] : 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int col0 = colh + c * 32;
                    // the exact sums first (debug output): stored after the dequant, they
                    // stayed live across it and pushed the epilogue into local memory
                    if (p.acc_out != nullptr && row_ok && col0 < p.n) {
                        int32_t *dst = p.acc_out + static_cast<int64_t>(row) * p.n + col0;
                        if (col0 + 32 <= p.n) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                reinterpret_cast<int4 *>(dst)[j] =
                                    make_int4(sum[c * 32 + 4 * j], sum[c * 32 + 4 * j + 1], sum[c * 32 + 4 * j + 2],
                                              sum[c * 32 + 4 * j + 3]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (col0 + i < p.n) dst[i] = sum[c * 32 + i];
                        }
                    }
                    uint32_t pk[16];
                    if (col0 + 32 <= p.n) {
                        // a whole chunk: its column scales and biases by 16-byte read-only
                        // loads (16-byte aligned: col0 % 32 == 0), 8 columns at a time (with the
                        // 128 running sums live, a group of 16 left too few registers)
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            const int cg = col0 + 8 * g;
                            float sc[8], bs[8];
#pragma unroll
                            for (int q4 = 0; q4 < 2; ++q4) {
                                const float4 t = __ldg(reinterpret_cast<const float4 *>(p.x2_scale + cg) + q4);
                                sc[4 * q4] = t.x;
                                sc[4 * q4 + 1] = t.y;
                                sc[4 * q4 + 2] = t.z;
                                sc[4 * q4 + 3] = t.w;
                            }
                            if (p.bias_q_bf16) {
                                const uint4 t = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.bias_q) + cg));
                                const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    bs[2 * e] = __uint_as_float(w[e] << 16);
                                    bs[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
                                }
                            } else {
#pragma unroll
                                for (int q4 = 0; q4 < 2; ++q4) {
                                    const float4 t =
                                        __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p.bias_q) + cg) + q4);
                                    bs[4 * q4] = t.x;
                                    bs[4 * q4 + 1] = t.y;
                                    bs[4 * q4 + 2] = t.z;
                                    bs[4 * q4 + 3] = t.w;
                                }
                            }
#pragma unroll
                            for (int i = 0; i < 8; i += 2) {
                                float o[2];
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    float v = __int2float_rn(sum[c * 32 + 8 * g + i + e]);
                                    v = __fmul_rn(v, s1);
                                    v = __fmul_rn(v, sc[i + e]);
                                    o[e] = __fadd_rn(v, bs[i + e]);
                                }
                                pk[4 * g + (i >> 1)] = pack2<true>(o[0], o[1]);
                            }
                        }
                    } else {
                        // the ragged last chunk: columns clamped to the output
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float o[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int col = min(col0 + i + e, p.n - 1);
                                float v = __int2float_rn(sum[c * 32 + i + e]);
                                v = __fmul_rn(v, s1);
                                v = __fmul_rn(v, p.x2_scale[col]);
                                const float bv = p.bias_q_bf16 ? load16<true>(p.bias_q, col)
                                                               : static_cast<const float *>(p.bias_q)[col];
                                o[e] = __fadd_rn(v, bv);
                            }
                            pk[i >> 1] = pack2<true>(o[0], o[1]);
                        }
                    }
                    put(c, pk);
                }
            }
        }
        // every output store has completed before the CTA can exit
        if constexpr (kTmaOut) {
            if (lane == 0) ptx::bulk_wait_group<0>();
            __syncwarp();
        }
    }

    __syncthreads();
    if constexpr (kPair) ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<kG>(tmem_base, kTmemCols);
    }
}

}  // namespace mc2
