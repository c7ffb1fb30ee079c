// gemm_tcgen05.cuh -- the fused MC2 GEMM for sm_103a.
//
// One persistent kernel serves both operations:
//   * AllGatherMatmul ("torch_npu.npu_all_gather_base_mm", 功能说明/输出说明):
//     A = concat_m of the per-rank chunks, read in place through one TMA
//     tensor map per chunk; out = A @ B (+ bias) rounded to bf16/fp16; the
//     gathered matrix is written from the A tiles already in shared memory
//     (one TMA store per (m-tile, k-tile), by the n-tile-0 tiles only).
//   * AlltoAllQuantMatmul ("aclnnAlltoAllQuantMatmul", 计算公式): A and B
//     hold int8 values as exact fp16; the fp32 tensor-core accumulator stays
//     exact while every partial sum is below 2^24, so the K loop is cut into
//     blocks of at most 1024 (1024 * 127 * 127 < 2^24) and each block's fp32
//     sum is flushed into an int32 register total; the epilogue then applies
//     the per-token x per-channel dequant and the bias in fp32 and rounds to bf16.
//
// Tile 128 x 256 x 64 (M x N x K), 16-bit operands in 128-byte-swizzled
// shared memory, 4-stage TMA ring, tcgen05.mma kind::f16 (M=128, N=256) into
// two 256-column TMEM accumulators so the epilogue of one tile (or K block)
// overlaps the MMAs of the next.
//
// Warp roles (384 threads):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator and MMA issuer (one lane)
//   warp 2      gathered-output TMA store (one lane; AllGather with gather only)
//   warp 3      idle
//   warps 4-11  epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (its rows) and
//               half (w-4)/4 of the 256 accumulator columns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace mc2 {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kMaxAMaps = 8;
constexpr int kNumEpiWarps = 8;
constexpr int kNumThreads = 128 + kNumEpiWarps * 32;
constexpr uint32_t kATileBytes = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kBTileBytes = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
constexpr uint32_t kTmemCols = 512;              // two 256-column fp32 accumulators
constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024 + 1024;
constexpr int kGroupM = 8;                       // m-tiles per raster group (L2 reuse of B)

enum AMode : int { A_SINGLE = 0, A_MCONCAT = 1, A_KINTERLEAVE = 2 };

struct GemmParams {
    CUtensorMap a_maps[kMaxAMaps];  // A operand: one map, or one per rank's chunk
    CUtensorMap b_map;              // B operand: (n, k) K-major or (k, n) N-major
    CUtensorMap g_map;              // gathered output (m, k), same box and swizzle as A
    int num_a_maps;
    int a_mode;
    int a_box_rows;                 // A_MCONCAT: rows per TMA box (divides m_local and kBM)
    int m, n, k;
    int m_local;                    // A_MCONCAT: rows per chunk
    int k_local;                    // A_KINTERLEAVE: columns per chunk
    int b_mn_major;
    int gather;
    int kblock_tiles;               // integer path: k-tiles per exact fp32 block
    void *out;                      // (m, n): dtype (float path) / bf16 (integer path)
    const void *bias16;             // float path: (n) in the operand dtype, or null
    const float *x1_scale;          // integer path: (m)
    const float *x2_scale;          // integer path: (n)
    const void *bias_q;             // integer path: (n) fp32 or bf16, or null
    int bias_q_bf16;
    int32_t *acc_out;               // integer path: optional (m, n)
    int *status;                    // device word set to -7 when a bounded wait gives up
    uint64_t wait_limit_ns;
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &mb, int &nb) {
    const int span = kGroupM * num_n;
    const int g = tile / span;
    const int first_m = g * kGroupM;
    const int gsz = min(num_m - first_m, kGroupM);
    const int r = tile - g * span;
    mb = first_m + r % gsz;
    nb = r / gsz;
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const GemmParams &p,
                                              volatile int *abort_flag) {
    if (*abort_flag) return false;
    if (ptx::mbar_wait(bar, parity, p.wait_limit_ns)) return true;
    *abort_flag = 1;
    if (p.status) atomicExch(p.status, -7);
    return false;
}

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

// Store 32 consecutive 16-bit outputs of one row (col0 .. col0+31), masked at n.
__device__ __forceinline__ void store_row32_16(void *out, int n, int row, int col0, const uint32_t (&pk)[16]) {
    uint16_t *dst = reinterpret_cast<uint16_t *>(out) + static_cast<int64_t>(row) * n + col0;
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

template <bool kBF16, bool kIntPath>
__global__ void __launch_bounds__(kNumThreads, 1) mc2_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *full_bar = bars;
    uint64_t *empty_bar = bars + kStages;
    uint64_t *tfull_bar = bars + 2 * kStages;
    uint64_t *tempty_bar = bars + 2 * kStages + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 4);
    __shared__ int abort_flag_s;
    volatile int *abort_flag = &abort_flag_s;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_m = (p.m + kBM - 1) / kBM;
    const int num_n = (p.n + kBN - 1) / kBN;
    const int num_tiles = num_m * num_n;
    const int num_k = (p.k + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        abort_flag_s = 0;
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), p.gather ? 2 : 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&tfull_bar[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&tempty_bar[b]), kNumEpiWarps);
        }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        for (int i = 0; i < p.num_a_maps; ++i) ptx::prefetch_tmap(&p.a_maps[i]);
        ptx::prefetch_tmap(&p.b_map);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t armed_phase[kStages];
        bool armed[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) armed[s] = false, armed_phase[s] = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, num_m, num_n, mb, nb);
            const int m0 = mb * kBM, n0 = nb * kBN;
            for (int kt = 0; kt < num_k; ++kt) {
                if (!wait_or_abort(ptx::smem_u32(&empty_bar[stage]), phase ^ 1u, p, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
                const uint32_t sA = ptx::smem_u32(smem + stage * kStageBytes);
                const uint32_t sB = sA + kATileBytes;
                ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                armed[stage] = true;
                armed_phase[stage] = phase;
                const int k0 = kt * kBK;
                if (p.a_mode == A_MCONCAT) {
                    const int nbox = kBM / p.a_box_rows;
                    for (int j = 0; j < nbox; ++j) {
                        const int i0 = m0 + j * p.a_box_rows;
                        const int c = min(i0 / p.m_local, p.num_a_maps - 1);
                        const int li = i0 - c * p.m_local;
                        ptx::tma_load_2d(sA + j * p.a_box_rows * 128, &p.a_maps[c], k0, li, fb);
                    }
                } else if (p.a_mode == A_KINTERLEAVE) {
                    const int c = k0 / p.k_local;
                    ptx::tma_load_2d(sA, &p.a_maps[c], k0 - c * p.k_local, m0, fb);
                } else {
                    ptx::tma_load_2d(sA, &p.a_maps[0], k0, m0, fb);
                }
                if (p.b_mn_major) {
#pragma unroll
                    for (int j = 0; j < kBN / 64; ++j) ptx::tma_load_2d(sB + j * (kBK * 128), &p.b_map, n0 + 64 * j, k0, fb);
                } else {
                    ptx::tma_load_2d(sB, &p.b_map, k0, n0, fb);
                }
                if (++stage == kStages) stage = 0, phase ^= 1u;
            }
        }
        if (!ok) {
            // let copies already in flight land before the CTA can exit
            for (int s = 0; s < kStages; ++s)
                if (armed[s]) (void)ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), armed_phase[s], p.wait_limit_ns);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = ptx::idesc_f16(kBF16 && !kIntPath, p.b_mn_major != 0, kBM, kBN);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t acc_iter = 0;
        bool ok = true;
        uint32_t d_tmem = tmem_base;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            for (int kt = 0; kt < num_k; ++kt) {
                const int kin = kIntPath ? (kt % p.kblock_tiles) : kt;  // k-tile index inside the block
                if (kin == 0) {
                    const uint32_t b = acc_iter & 1u;
                    if (!wait_or_abort(ptx::smem_u32(&tempty_bar[b]), ((acc_iter >> 1) & 1u) ^ 1u, p, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    d_tmem = tmem_base + b * kBN;
                }
                if (!wait_or_abort(ptx::smem_u32(&full_bar[stage]), phase, p, abort_flag)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sA = ptx::smem_u32(smem + stage * kStageBytes);
                const uint32_t sB = sA + kATileBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = ptx::smem_desc_sw128(sA + kk * 32, 16, 1024);
                    const uint64_t bd = p.b_mn_major ? ptx::smem_desc_sw128(sB + kk * 2048, kBK * 128, 1024)
                                                     : ptx::smem_desc_sw128(sB + kk * 32, 16, 1024);
                    ptx::mma_f16_ss(d_tmem, ad, bd, idesc, (kin > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
                if (++stage == kStages) stage = 0, phase ^= 1u;
                const bool block_end = kIntPath ? (kin == p.kblock_tiles - 1 || kt == num_k - 1) : (kt == num_k - 1);
                if (block_end) {
                    ptx::mma_commit(ptx::smem_u32(&tfull_bar[acc_iter & 1u]));
                    ++acc_iter;
                }
            }
        }
    } else if (warp == 2 && lane == 0 && p.gather) {
        // ------------------------------------------------------------ gathered store
        ptx::prefetch_tmap(&p.g_map);
        int stage = 0;
        uint32_t phase = 0;
        int pending_stage = -1;  // stage whose store may still be reading smem
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, num_m, num_n, mb, nb);
            bool ok = true;
            for (int kt = 0; kt < num_k; ++kt) {
                if (!wait_or_abort(ptx::smem_u32(&full_bar[stage]), phase, p, abort_flag)) {
                    ok = false;
                    break;
                }
                if (nb == 0) {
                    const uint32_t sA = ptx::smem_u32(smem + stage * kStageBytes);
                    ptx::tma_store_2d(&p.g_map, kt * kBK, mb * kBM, sA);
                    ptx::bulk_commit_group();
                    // release the previous stage once its store has finished reading
                    ptx::bulk_wait_group_read<1>();
                    if (pending_stage >= 0) ptx::mbar_arrive(ptx::smem_u32(&empty_bar[pending_stage]));
                    pending_stage = stage;
                } else {
                    if (pending_stage >= 0) {
                        ptx::bulk_wait_group_read<0>();
                        ptx::mbar_arrive(ptx::smem_u32(&empty_bar[pending_stage]));
                        pending_stage = -1;
                    }
                    ptx::mbar_arrive(ptx::smem_u32(&empty_bar[stage]));
                }
                if (++stage == kStages) stage = 0, phase ^= 1u;
            }
            if (!ok) break;
        }
        ptx::bulk_wait_group_read<0>();
        if (pending_stage >= 0) ptx::mbar_arrive(ptx::smem_u32(&empty_bar[pending_stage]));
        ptx::bulk_wait_group<0>();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quadrant this warp may access
        const int half = (warp - 4) >> 2;     // which 128 of the 256 columns
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        uint32_t acc_iter = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, num_m, num_n, mb, nb);
            const int row = mb * kBM + 32 * q + lane;
            const int colh = nb * kBN + half * 128;
            bool ok = true;
            if constexpr (!kIntPath) {
                const uint32_t b = acc_iter & 1u;
                if (!wait_or_abort(ptx::smem_u32(&tfull_bar[b]), (acc_iter >> 1) & 1u, p, abort_flag)) break;
                ptx::tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const int col0 = colh + c * 32;
                    if (col0 >= p.n) break;
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(tmem_base + lane_addr + b * kBN + half * 128 + c * 32, r);
                    ptx::tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    if (p.bias16 != nullptr) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col0 + i < p.n) v[i] = __fadd_rn(v[i], load16<kBF16>(p.bias16, col0 + i));
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) pk[i] = pack2<kBF16>(v[2 * i], v[2 * i + 1]);
                    if (row < p.m) store_row32_16(p.out, p.n, row, col0, pk);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&tempty_bar[b]));
                ++acc_iter;
            } else {
                int32_t sum[128];
#pragma unroll
                for (int i = 0; i < 128; ++i) sum[i] = 0;
                const int nkb = (num_k + p.kblock_tiles - 1) / p.kblock_tiles;
                for (int kb = 0; kb < nkb; ++kb) {
                    const uint32_t b = acc_iter & 1u;
                    if (!wait_or_abort(ptx::smem_u32(&tfull_bar[b]), (acc_iter >> 1) & 1u, p, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (colh + c * 32 < p.n) {
                            uint32_t r[32];
                            ptx::tmem_ld_32x32b_x32(tmem_base + lane_addr + b * kBN + half * 128 + c * 32, r);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i) sum[c * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
                        }
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&tempty_bar[b]));
                    ++acc_iter;
                }
                if (!ok) break;
                const float s1 = row < p.m ? p.x1_scale[row] : 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int col0 = colh + c * 32;
                    if (col0 < p.n && row < p.m) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float o[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int col = min(col0 + i + e, p.n - 1);
                                float v = __int2float_rn(sum[c * 32 + i + e]);
                                v = __fmul_rn(v, s1);
                                v = __fmul_rn(v, p.x2_scale[col]);
                                if (p.bias_q != nullptr) {
                                    const float bv = p.bias_q_bf16 ? load16<true>(p.bias_q, col)
                                                                   : reinterpret_cast<const float *>(p.bias_q)[col];
                                    v = __fadd_rn(v, bv);
                                }
                                o[e] = v;
                            }
                            pk[i >> 1] = pack2<true>(o[0], o[1]);
                        }
                        store_row32_16(p.out, p.n, row, col0, pk);
                        if (p.acc_out != nullptr) {
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
                    }
                }
            }
            if (!ok) break;
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace mc2
