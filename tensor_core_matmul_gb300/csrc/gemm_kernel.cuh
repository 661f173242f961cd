// Persistent, warp-specialised bf16 GEMM for sm_103a:
//   C[M x N] (column-major) = alpha * A[M x K] (row-major) * B[K x N] (column-major)
//                             + beta * C
// with fp32 accumulation in tensor memory.
//
// Structure, following the H100 work log "在 H100 上超越 cuBLAS：一份工作日志" and
// re-designed for Blackwell:
//  * "内核 4：隐藏加载延迟": a producer feeds a circular shared-memory queue
//    guarded by full/empty barriers; here the producer is one thread of warp 0
//    issuing TMA tile loads (128-byte swizzle, as chosen in the retelling
//    "Hopper H100 GEMM优化实战", section 2.2).
//  * "内核 5": the register-file accumulator limit that forced two consumer
//    warpgroups on Hopper is gone: one thread of warp 1 issues tcgen05.mma and
//    the fp32 accumulator lives in TMEM (128 lanes x BN columns).
//  * "内核 6：隐藏存储延迟": persistent CTAs (one per SM, or one pair per two
//    SMs) walk a grouped tile order; two TMEM accumulators let the epilogue of
//    tile i overlap the mainloop of tile i+1.
//  * "内核 7：更快的屏障": phase-parity mbarriers; tcgen05.commit arrives on
//    the empty barrier of a stage once the MMAs that read it are done.
//  * "内核 8：线程块集群": a cluster of 2 CTAs shares one tile.  On Blackwell
//    the pair runs a single cta_group::2 MMA of M = 256: each CTA loads its own
//    128 rows of A and its own half of the B tile, and the MMA reads both
//    CTAs' shared memory, so no operand is fetched twice inside the pair.
//  * "内核 9：微优化": the first MMA of a tile does not accumulate (enable-input-d
//    false), which replaces zeroing the accumulator.
//  * Edge tiles (the "DeepGEMM" article, sections 4.2-4.3): TMA fills
//    out-of-range A/B elements with zeros, so they add nothing; the epilogue
//    masks out-of-range rows and columns of C.
//
// Every wait on a barrier is bounded by %globaltimer.  On expiry the waiting
// thread records TCGEMM_ERR_TIMEOUT in the device status word, raises the
// CTA's abort flag and leaves its loop; the CTA then drains its own copies and
// MMAs (again with bounded waits), frees its TMEM and exits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace tcg {

// Device status word: [0] = error code (0 = none), [1] = where, [2] = block.
__device__ uint32_t g_tcgemm_status[4];

enum : uint32_t {
    kWhereProducer = 1,
    kWhereMma = 2,
    kWhereEpilogue = 3,
    kWhereDrain = 4,
    kWhereSelfTest = 5,
};

constexpr uint32_t kStatusTimeout = 5;  // TCGEMM_ERR_TIMEOUT

__device__ __forceinline__ void raise_timeout(uint32_t where) {
    if (atomicCAS(&g_tcgemm_status[0], 0u, kStatusTimeout) == 0u) {
        g_tcgemm_status[1] = where;
        g_tcgemm_status[2] = blockIdx.x;
    }
    __threadfence();
}

struct WaitCtx {
    volatile uint32_t* abort;  // CTA-wide abort flag in shared memory
    uint64_t timeout_ns;
};

// Bounded wait for the phase with the given parity.  Returns false (after
// recording a timeout, or seeing another thread's abort) if it gave up.
template <bool kClusterScope>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                           uint32_t where) {
    auto probe = [&]() {
        return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (probe()) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (probe()) return true;
        if ((n & 15u) == 0u) {
            if (*w.abort) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                raise_timeout(where);
                *w.abort = 1u;
                return false;
            }
        }
    }
}

// ------------------------------------------------------------ scheduling --

// Tile order over the tiles_m x tiles_n grid of output tiles.  Consecutive
// indices run down a band of `group_m` tile-rows before moving one tile-column
// right, so the tiles that the persistent CTAs work on at the same time share
// rows of A and columns of B in L2 (the work log's "调度与 L2 缓存").
__host__ __device__ __forceinline__ void grouped_tile(int t, int tiles_m, int tiles_n, int group_m,
                                                      int& tm, int& tn) {
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int rows = (tiles_m - first_m) < group_m ? (tiles_m - first_m) : group_m;
    const int r = t - g * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

struct GemmParams {
    int M, N, K;
    int tiles_m, tiles_n, num_kb, group_m;
    int64_t ldc;
    void* C;
    float alpha, beta;
    uint64_t timeout_ns;
};

template <int CTA_GROUP, int BN, int STAGES>
struct GemmCfg {
    static constexpr int kBK = 64;                        // 64 bf16 = one 128-byte swizzle row
    static constexpr int kRowsA = 128;                    // A rows per CTA
    static constexpr int kBM = 128 * CTA_GROUP;           // MMA M (pair tile height)
    static constexpr int kRowsB = BN / CTA_GROUP;         // B rows (tile columns) per CTA
    static constexpr int kUmmaK = 16;
    static constexpr uint32_t kABytes = kRowsA * kBK * 2;
    static constexpr uint32_t kBBytes = kRowsB * kBK * 2;
    static constexpr uint32_t kStageTx = CTA_GROUP * (kABytes + kBBytes);  // bytes landing per stage
    static constexpr uint32_t kTmemCols = 2 * BN;         // two accumulators
    static constexpr int kThreads = 192;                  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
    static constexpr uint32_t kBarOff = STAGES * (kABytes + kBBytes);
    static constexpr uint32_t kNumBars = 2 * STAGES + 4 + 1;
    static constexpr uint32_t kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;  // + alignment slack
    static_assert(kTmemCols <= 512, "TMEM has 512 columns");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "epilogue works in 32-column chunks");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
};

template <typename OutT>
__device__ __forceinline__ float load_out(const OutT* p);
template <>
__device__ __forceinline__ float load_out<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_out<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename OutT>
__device__ __forceinline__ void store_out(OutT* p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

template <int CTA_GROUP, int BN, int STAGES, typename OutT>
__global__ void __launch_bounds__(192, 1)
    gemm_bf16_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmParams p) {
    using Cfg = GemmCfg<CTA_GROUP, BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];

    // 1 KB-aligned carve-up: [A stages][B stages][barriers][tmem slot][abort]
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_u32);
    const uint32_t sA0 = base;
    const uint32_t sB0 = base + STAGES * Cfg::kABytes;
    const uint32_t bar0 = base + Cfg::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kBarOff + Cfg::kNumBars * 8);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t rank = (CTA_GROUP == 2) ? cluster_ctarank() : 0u;
    const int cluster_id = blockIdx.x / CTA_GROUP;
    const int num_clusters = gridDim.x / CTA_GROUP;
    const int num_tiles = p.tiles_m * p.tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4 * CTA_GROUP);  // one arrive per epilogue warp of each CTA
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc<CTA_GROUP>(smem_u32(tmem_slot), Cfg::kTmemCols);
    tc_fence_before_sync();
    if constexpr (CTA_GROUP == 1) {
        __syncthreads();
    } else {
        cluster_sync();
    }
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtx wctx{abort_flag, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            uint32_t stage = 0, phase = 0;
            uint64_t issued = 0;
            bool ok = true;
            for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
                int tm, tn;
                grouped_tile(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                const int a_row = tm * Cfg::kBM + static_cast<int>(rank) * Cfg::kRowsA;
                const int b_row = tn * BN + static_cast<int>(rank) * Cfg::kRowsB;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_phase<false>(empty_bar(stage), phase ^ 1u, wctx, kWhereProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sA0 + stage * Cfg::kABytes;
                    const uint32_t sb = sB0 + stage * Cfg::kBBytes;
                    if constexpr (CTA_GROUP == 1) {
                        mbar_arrive_expect_tx(full_bar(stage), Cfg::kStageTx);
                        tma_load_2d(sa, &tmA, full_bar(stage), kb * Cfg::kBK, a_row);
                        tma_load_2d(sb, &tmB, full_bar(stage), kb * Cfg::kBK, b_row);
                    } else {
                        // Both CTAs' bytes land on the leader's barrier.
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), Cfg::kStageTx);
                        const uint32_t fb = map_to_cta(full_bar(stage), 0);
                        tma_load_2d_pair(sa, &tmA, fb, kb * Cfg::kBK, a_row);
                        tma_load_2d_pair(sb, &tmB, fb, kb * Cfg::kBK, b_row);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Drain: every load this thread issued has landed before the CTA
            // may exit.  The leader (or a lone CTA) sees that on its full
            // barriers; a pair's second CTA sees it when the leader's MMA
            // frees the stage again.
            for (int s = 0; s < STAGES; ++s) {
                if (issued <= static_cast<uint64_t>(s)) break;
                const uint64_t times = (issued - s - 1) / STAGES + 1;
                const uint32_t par = static_cast<uint32_t>((times - 1) & 1u);
                if (CTA_GROUP == 1 || rank == 0) {
                    wait_phase<false>(full_bar(s), par, wctx, kWhereDrain);
                } else {
                    wait_phase<false>(empty_bar(s), par, wctx, kWhereDrain);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0 && (CTA_GROUP == 1 || rank == 0)) {
            constexpr uint32_t kIdesc = idesc_bf16_f32(Cfg::kBM, BN);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
                if (!wait_phase<CTA_GROUP == 2>(tempty_bar(acc), acc_phase ^ 1u, wctx, kWhereMma)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_phase<false>(full_bar(stage), phase, wctx, kWhereMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t ad = sdesc_kmajor_sw128(sA0 + stage * Cfg::kABytes);
                    const uint64_t bd = sdesc_kmajor_sw128(sB0 + stage * Cfg::kBBytes);
#pragma unroll
                    for (int k = 0; k < Cfg::kBK / Cfg::kUmmaK; ++k) {
                        // +32 bytes along K per step: (32 >> 4) = 2 in the address field.
                        mma_bf16<CTA_GROUP>(d_tmem, ad + 2u * k, bd + 2u * k, kIdesc,
                                            (kb | k) != 0 ? 1u : 0u);
                    }
                    if constexpr (CTA_GROUP == 1) {
                        mma_commit(empty_bar(stage));
                    } else {
                        mma_commit_pair(empty_bar(stage), 0x3);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (CTA_GROUP == 1) {
                    mma_commit(tfull_bar(acc));
                } else {
                    mma_commit_pair(tfull_bar(acc), 0x3);
                }
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Drain: all MMAs issued by this thread have completed.
            if constexpr (CTA_GROUP == 1) {
                mma_commit(drain_bar);
            } else {
                mma_commit_pair(drain_bar, 0x1);
            }
            wait_phase<false>(drain_bar, 0, wctx, kWhereDrain);
        }
    } else {
        // --------------------------------------------------- epilogue --
        // Warp w may only touch TMEM lanes 32*(w%4) .. 32*(w%4)+31.
        const uint32_t q = warp & 3u;
        OutT* C = static_cast<OutT*>(p.C);
        const bool has_beta = p.beta != 0.0f;
        uint32_t acc = 0, acc_phase = 0;
        for (int t = cluster_id; t < num_tiles; t += num_clusters) {
            int tm, tn;
            grouped_tile(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            uint32_t ok = 1;
            if (lane == 0) ok = wait_phase<false>(tfull_bar(acc), acc_phase, wctx, kWhereEpilogue) ? 1u : 0u;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            const int64_t row = static_cast<int64_t>(tm) * Cfg::kBM + rank * 128 + q * 32 + lane;
            const bool row_ok = row < p.M;
            const uint32_t tbase = tmem_base + ((q * 32u) << 16) + acc * BN;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                const int64_t col0 = static_cast<int64_t>(tn) * BN + c;
                if (col0 >= p.N) break;
                uint32_t r[32];
                tmem_ld32(tbase + c, r);
                tmem_ld_wait32(r);
                if (row_ok) {
                    OutT* dst = C + col0 * p.ldc + row;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (col0 + j < p.N) {
                            float v = __uint_as_float(r[j]);
                            if (has_beta) {
                                v = fmaf(p.alpha, v, p.beta * load_out<OutT>(dst));
                            } else {
                                v = p.alpha * v;
                            }
                            store_out<OutT>(dst, v);
                        }
                        dst += p.ldc;
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CTA_GROUP == 1) {
                    mbar_arrive(tempty_bar(acc));
                } else {
                    mbar_arrive_cluster(map_to_cta(tempty_bar(acc), 0));
                }
            }
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    // ------------------------------------------------------- teardown --
    __syncwarp();
    tc_fence_before_sync();
    if constexpr (CTA_GROUP == 1) {
        __syncthreads();
    } else {
        cluster_sync();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CTA_GROUP>(tmem_base, Cfg::kTmemCols);
    }
}

// C = beta * C (or 0 when beta == 0): the K == 0 case, where the product is
// an empty sum.
template <typename OutT>
__global__ void scale_c_kernel(OutT* C, int64_t M, int64_t N, int64_t ldc, float beta) {
    const int64_t total = M * N;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = idx / M, i = idx - j * M;
        OutT* dst = C + j * ldc + i;
        store_out<OutT>(dst, beta == 0.0f ? 0.0f : beta * load_out<OutT>(dst));
    }
}

// Self test of the bounded wait: one thread waits on a barrier that nothing
// ever arrives on, gives up after `timeout_ns` and records the timeout in the
// status word.  No TMA, no TMEM, no MMA.
__global__ void selftest_wait_kernel(uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx w{&abort_flag, timeout_ns};
        (void)wait_phase<false>(smem_u32(&bar), 0, w, kWhereSelfTest);
    }
    __syncthreads();
}

}  // namespace tcg
