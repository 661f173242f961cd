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
// Stream-K (not on the pages; the work log's conclusion attributes its
// remaining per-size gaps to tuning).  When there are too few tiles to keep
// the persistent clusters busy (the host decides; see use_stream_k), the tiles
// of the last, partial round are not handed out whole: their k-blocks, taken
// in order, are cut into one contiguous range per cluster, so every cluster
// does the same amount of that work.  A range that covers only part of a tile produces an fp32 partial
// tile, written through TMA to the cluster's workspace slot; a second, small
// kernel (sk_reduce_kernel) then adds each shared tile's partials in K order
// and runs its epilogue.  No CTA ever waits for another.
//
// Every wait on a barrier is bounded by %globaltimer.  On expiry the waiting
// thread records TCGEMM_ERR_TIMEOUT in the device status word, raises the
// CTA's abort flag and leaves its loop; the CTA then drains its own copies and
// MMAs (again with bounded waits), frees its TMEM and exits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include <type_traits>

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

// Cell d of the Hilbert curve over a 2^order x 2^order grid (the iterative
// form that consumes d two bits at a time, lowest first, reflecting and
// transposing the partial coordinates at each level).  The curve starts at
// (0, 0) and ends at (2^order - 1, 0).
__host__ __device__ __forceinline__ void hilbert_d2xy(int order, int d, int& x, int& y) {
    x = 0;
    y = 0;
    for (int s = 1; s < (1 << order); s <<= 1) {
        const int rx = 1 & (d >> 1);
        const int ry = 1 & (d ^ rx);
        if (ry == 0) {
            if (rx == 1) {
                x = s - 1 - x;
                y = s - 1 - y;
            }
            const int t = x;
            x = y;
            y = t;
        }
        x += s * rx;
        y += s * ry;
        d >>= 2;
    }
}

// Tile order of the H100 work log's "内核 11：希尔伯特曲线": the tiles of the
// tiles_m x tiles_n grid in the order in which the Hilbert curve of the
// enclosing 2^order square visits them, cells outside the grid skipped.  The
// t-th tile is found from the top down: the curve covers the aligned
// quarter-squares in the order the coarser curve visits its cells, so at
// each level the child that holds the t-th tile is the first whose running
// count of in-grid cells exceeds t.  Consecutive indices are neighbouring
// tiles, so the tiles the persistent CTAs work on at once form a compact
// patch (rows of A and columns of B shared in L2), and the next round's
// patch borders it.
__host__ __device__ __forceinline__ void hilbert_tile(int t, int tiles_m, int tiles_n, int order, int& tm, int& tn) {
    int q = 0;
    for (int j = order - 1; j >= 0; --j) {
        const int side = 1 << j;
        for (int c = 0; c < 4; ++c) {
            int x, y;
            hilbert_d2xy(order - j, 4 * q + c, x, y);
            const int w = min(max(tiles_m - (x << j), 0), side);
            const int h = min(max(tiles_n - (y << j), 0), side);
            if (t < w * h || c == 3) {
                q = 4 * q + c;
                break;
            }
            t -= w * h;
        }
    }
    hilbert_d2xy(order, q, tm, tn);
}

struct GemmParams {
    int M, N, K;
    int tiles_m, tiles_n, num_kb, group_m;
    int hilbert;         // 0: grouped band order; else the Hilbert order over a 2^hilbert square
    int grid_m, grid_n;  // grid of tiles the unit order walks
    int tiles_dp;        // tiles computed whole, round-robin over the clusters
    int sk_tiles;        // trailing tiles whose k-blocks are shared out by stream-K (0: none)
    int64_t sk_iters;    // sk_tiles * num_kb
    int64_t ldc;
    void* C;
    float alpha, beta;
    int in_fmt;          // 8-bit operands: bit 0 the MMA's A operand, bit 1 its B operand: 0 = E4M3, 1 = E5M2
    int a_mn, b_mn;      // MMA operand A / B stored MN-major (M or N contiguous; bf16 only)
    // Fused epilogue: out = act(alpha*acc + beta*C + bias[column of C]).
    const void* bias;    // one value per column of C (per row of D in the transposed product), or null
    int bias_kind;       // 0 none, 1 fp32, 2 bf16
    int act;             // kAct*
    // int8 output: code = saturate(rne(fmaf(value, qscale[row of C], qzero))).
    const float* qscale;
    float qzero;
    // Transposed product on CTA pairs: rows of the MMA's A operand (columns
    // of C) loaded per CTA, a multiple of 8 up to the stage's capacity; a
    // pair's tile is 2 * rows_a rows of D.  Unused by the other kernels.
    int rows_a;
    uint64_t timeout_ns;
    // Self test of the give-up path (tcgemm_selftest_withheld_load): the
    // producer of CTA 0 withholds the arrival and the loads of its k-block
    // number `withhold_kb` (-1: never), so that the MMA's wait for it runs
    // out.
    int withhold_kb;
};

// The tile of unit index t under the launch's visiting order.
__host__ __device__ __forceinline__ void unit_tile_of(const GemmParams& p, int t, int& tm, int& tn) {
    if (p.hilbert > 0) {
        hilbert_tile(t, p.grid_m, p.grid_n, p.hilbert, tm, tn);
    } else {
        grouped_tile(t, p.grid_m, p.grid_n, p.group_m, tm, tn);
    }
}

// ------------------------------------------------------ fused epilogue --
// The "DeepGEMM" article (section 6.1) fuses the bias add and the ReLU/GELU
// that follow a fully connected layer into the GEMM's epilogue; the order is
// bias, then activation, then the store.  Both run in fp32 on the value
// alpha*acc (+ beta*C); the activation is chosen per call (a warp-uniform
// branch) rather than per compiled kernel.
//
// The epilogue warps share the SM sub-partitions' issue slots with the TMA
// and MMA warps of the next tile's mainloop, so the activations are written
// to issue few instructions: no data-dependent branches, and pairs of values
// through Blackwell's packed fp32x2 operations (__ffma2_rn and friends,
// IEEE-rounded per lane, so a pair gives the same bits as two scalar calls).
enum : int { kActNone = 0, kActRelu = 1, kActGelu = 2, kActGeluTanh = 3 };

// P(t) of erfc(z) = t * exp(-z^2 + P(t)), t = 1/(1 + z/2), z >= 0: the form of
// Press et al., "Numerical Recipes" (2nd ed., section 6.2); coefficients (of
// t^0 .. t^9) from the least-squares Chebyshev fit in fit_erfc.py beside this
// file (relative error of erfc below 1.1e-7 on [0, 30] in exact arithmetic).
__device__ constexpr float kErfcP[10] = {-1.2655122f, 1.0000237f, 0.37409195f, 0.09678419f, -0.18628806f,
                                         0.27886808f, -1.135204f, 1.4885159f, -0.82215226f, 0.17087278f};
constexpr float kRsqrt2 = 0.70710678118654752f;        // 1/sqrt(2)
constexpr float kSqrt2OverPi = 0.79788456080286536f;   // sqrt(2/pi)
constexpr float kGeluCubic = 0.044715f;                 // the tanh approximation's cubic coefficient

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// GELU(x) = x * Phi(x), Phi(x) = erfc(-x/sqrt 2)/2, which is h = erfc(|x|/sqrt 2)/2
// for x < 0 and 1 - h for x >= 0 (no cancellation on either side).
__device__ __forceinline__ float2 gelu_erf2(float2 x) {
    const float2 w = __fmul2_rn(make_float2(fabsf(x.x), fabsf(x.y)), f2(kRsqrt2));
    const float2 d = __ffma2_rn(f2(0.5f), w, f2(1.0f));
    const float2 t = make_float2(__fdividef(1.0f, d.x), __fdividef(1.0f, d.y));
    float2 q = f2(kErfcP[9]);
#pragma unroll
    for (int k = 8; k >= 0; --k) q = __ffma2_rn(q, t, f2(kErfcP[k]));
    const float2 a = __ffma2_rn(make_float2(-w.x, -w.y), w, q);
    const float2 h = __fmul2_rn(__fmul2_rn(f2(0.5f), t), make_float2(__expf(a.x), __expf(a.y)));
    return __fmul2_rn(x, make_float2(x.x >= 0.0f ? 1.0f - h.x : h.x, x.y >= 0.0f ? 1.0f - h.y : h.y));
}

// x/2 (1 + tanh z) = x * sigmoid(2z), z = sqrt(2/pi) (x + 0.044715 x^3); with
// u = exp(-2|z|) <= 1, sigmoid(2z) = 1/(1+u) for z >= 0 and u/(1+u) below, so
// nothing overflows.
__device__ __forceinline__ float2 gelu_tanh2(float2 x) {
    const float2 k = __fmul2_rn(__fmul2_rn(x, x), f2(kGeluCubic));
    const float2 z = __fmul2_rn(__ffma2_rn(k, x, x), f2(kSqrt2OverPi));
    const float2 u = make_float2(__expf(-2.0f * fabsf(z.x)), __expf(-2.0f * fabsf(z.y)));
    const float2 den = __fadd2_rn(u, f2(1.0f));
    const float2 num = make_float2(z.x >= 0.0f ? 1.0f : u.x, z.y >= 0.0f ? 1.0f : u.y);
    return __fmul2_rn(x, make_float2(__fdividef(num.x, den.x), __fdividef(num.y, den.y)));
}

__device__ __forceinline__ float relu(float x) { return (x > 0.0f || x != x) ? x : 0.0f; }

__device__ __forceinline__ float2 activation2(float2 v, int act) {
    if (act == kActRelu) return make_float2(relu(v.x), relu(v.y));
    if (act == kActGelu) return gelu_erf2(v);
    if (act == kActGeluTanh) return gelu_tanh2(v);
    return v;
}

// One value: the same operations (a pair with a duplicate), so every path
// gives the same bits for the same input.
__device__ __forceinline__ float activation(float x, int act) { return activation2(f2(x), act).x; }

// In place on an even number of values held in registers.  The (warp-
// uniform) choice of activation is taken once, outside the loops, so that no
// code path computes an activation it does not return.
template <int W>
__device__ __forceinline__ void activation_n(float (&v)[W], int act) {
    static_assert(W % 2 == 0, "pairs");
    if (act == kActRelu) {
#pragma unroll
        for (int j = 0; j < W; ++j) v[j] = relu(v[j]);
    } else if (act == kActGelu) {
#pragma unroll
        for (int j = 0; j < W; j += 2) {
            const float2 r = gelu_erf2(make_float2(v[j], v[j + 1]));
            v[j] = r.x;
            v[j + 1] = r.y;
        }
    } else if (act == kActGeluTanh) {
#pragma unroll
        for (int j = 0; j < W; j += 2) {
            const float2 r = gelu_tanh2(make_float2(v[j], v[j + 1]));
            v[j] = r.x;
            v[j + 1] = r.y;
        }
    }
}

__device__ __forceinline__ float bias_at(const GemmParams& p, int64_t i) {
    if (p.bias_kind == 1) return __ldg(static_cast<const float*>(p.bias) + i);
    if (p.bias_kind == 2) return __bfloat162float(__ldg(static_cast<const __nv_bfloat16*>(p.bias) + i));
    return 0.0f;
}

__device__ __forceinline__ bool has_epilogue(const GemmParams& p) { return p.bias_kind != 0 || p.act != kActNone; }

// First stream-K iteration of cluster c: the ranges are [lo(c), lo(c+1)).
__host__ __device__ __forceinline__ int64_t sk_lo(int64_t c, int64_t iters, int64_t clusters) {
    return (c * iters) / clusters;
}

// The cluster whose range holds iteration `it` (the largest c with lo(c) <= it).
__host__ __device__ __forceinline__ int sk_owner(int64_t it, int64_t iters, int64_t clusters) {
    return static_cast<int>(((it + 1) * clusters - 1) / iters);
}

// Workspace slot of cluster c's piece of the stream-K tile starting at
// iteration t_begin: a cluster has at most two partial pieces, the first and
// the last segment of its range.
__host__ __device__ __forceinline__ int sk_slot(int c, int64_t t_begin, int64_t iters, int64_t clusters) {
    return 2 * c + (sk_lo(c, iters, clusters) >= t_begin ? 0 : 1);
}

// One unit of work for a cluster: a whole tile, or one piece of a stream-K tile.
struct WorkUnit {
    int tile;          // unit index in grouped order
    int kb0, kb1;      // k-block range [kb0, kb1)
    int slot;          // -1: a whole tile; else this piece's workspace slot
    int sk_tile;       // index among the stream-K tiles (-1 for round-robin tiles)
    int piece, npieces;  // place of this piece among the tile's pieces (K order)
};

// Walks the units of one cluster: first the segments of its stream-K range,
// then its share of the whole tiles.  Doing the shared tiles first lets the
// piece that finishes a shared tile last add up the partials in its epilogue
// warps while its MMA thread already works on whole tiles.  Producer, MMA and
// epilogue roles each run their own copy and see the same sequence.
struct UnitIter {
    int next_dp;   // next whole tile
    int stride;    // number of clusters
    int cluster;
    int64_t sk_it, sk_end;

    __host__ __device__ UnitIter(int cluster_id, int num_clusters)
        : next_dp(cluster_id), stride(num_clusters), cluster(cluster_id), sk_it(0), sk_end(0) {}

    // Must be called once with the launch parameters before next().
    __host__ __device__ void start(const GemmParams& p) {
        if (p.sk_tiles > 0) {
            sk_it = sk_lo(cluster, p.sk_iters, stride);
            sk_end = sk_lo(cluster + 1, p.sk_iters, stride);
        }
    }

    __host__ __device__ bool next(const GemmParams& p, WorkUnit& u) {
        if (sk_it < sk_end) {
            const int t = static_cast<int>(sk_it / p.num_kb);
            const int64_t t_begin = static_cast<int64_t>(t) * p.num_kb;
            const int64_t t_end = t_begin + p.num_kb;
            const int64_t seg_end = sk_end < t_end ? sk_end : t_end;
            u.tile = p.tiles_dp + t;
            u.sk_tile = t;
            u.kb0 = static_cast<int>(sk_it - t_begin);
            u.kb1 = static_cast<int>(seg_end - t_begin);
            if (u.kb0 == 0 && u.kb1 == p.num_kb) {
                u.slot = -1;
                u.piece = 0;
                u.npieces = 1;
            } else {
                const int first = sk_owner(t_begin, p.sk_iters, stride);
                const int last = sk_owner(t_end - 1, p.sk_iters, stride);
                u.piece = cluster - first;
                u.npieces = last - first + 1;
                u.slot = sk_slot(cluster, t_begin, p.sk_iters, stride);
            }
            sk_it = seg_end;
            return true;
        }
        if (next_dp < p.tiles_dp) {
            u.tile = next_dp;
            u.kb0 = 0;
            u.kb1 = p.num_kb;
            u.slot = -1;
            u.sk_tile = -1;
            u.piece = 0;
            u.npieces = 1;
            next_dp += stride;
            return true;
        }
        return false;
    }
};

// AROWS = 64 (single CTA, M <= 64 only): only the 64 real rows of A are
// loaded; the MMA still computes 128 rows and reads rows 64..127 from the
// shared memory that follows the A stage.  Those accumulator rows are never
// stored, so whatever they hold does not matter, and A's traffic halves.
// IN = 0: bf16 operands; IN = 1: 8-bit float operands (E4M3 or E5M2).  A
// k-block is one 128-byte swizzle row either way: 64 bf16 or 128 FP8 values.
template <int CTA_GROUP, int BN, int STAGES, int AROWS = 128, int IN = 0, int KS = 1>
struct GemmCfg {
    static constexpr int kInBytes = IN == 1 ? 1 : 2;       // bytes per operand element
    static constexpr int kBK = 128 / kInBytes;             // elements per k-block (one 128-byte row)
    static constexpr int kRowsA = AROWS;                  // A rows loaded per CTA
    static constexpr int kBM = 128 * CTA_GROUP;           // MMA M (pair tile height)
    static constexpr int kRowsB = BN / CTA_GROUP;         // B rows (tile columns) per CTA
    static constexpr int kUmmaK = 32 / kInBytes;           // K of one MMA instruction (32 bytes)
    static constexpr uint32_t kABytes = kRowsA * 128;
    static constexpr uint32_t kBBytes = kRowsB * 128;
    static constexpr uint32_t kStageTx = CTA_GROUP * (kABytes + kBBytes);  // bytes landing per stage
    static constexpr uint32_t kTmemCols = 2 * BN;         // two accumulators
    static constexpr uint32_t kTmemAlloc = kTmemCols <= 32 ? 32 : kTmemCols <= 64 ? 64 : kTmemCols <= 128 ? 128
                                         : kTmemCols <= 256 ? 256 : 512;  // allocations are powers of two
    static constexpr int kThreads = 192;                  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
    // Epilogue staging shared by the four epilogue warps: two buffers of one
    // 128-row x 32-column chunk of C (sized for fp32 output).
    static constexpr uint32_t kEpiBufBytes = 128 * 32 * 4;
    static constexpr uint32_t kEpiOff = STAGES * (kABytes + kBBytes);
    // A K-split cluster (KS = 2) also stages half an fp32 tile there for the peer.
    static constexpr uint32_t kEpiBytes = (KS == 2 && 128u * (BN / 2) * 4u > 2 * kEpiBufBytes) ? 128u * (BN / 2) * 4u
                                                                                               : 2 * kEpiBufBytes;
    static constexpr uint32_t kBarOff = kEpiOff + kEpiBytes;
    // full/empty per stage, tfull/tempty x 2, drain, C chunk loads (2 per
    // epilogue warp), xfull/xfree.
    static constexpr uint32_t kNumBars = 2 * STAGES + 4 + 1 + 8 + 2;
    // The fused epilogue's bias values for the current tile's BN columns
    // (fp32), staged once per tile.
    static constexpr uint32_t kBiasOff = (kBarOff + kNumBars * 8 + 16 + 15) / 16 * 16;
    static constexpr uint32_t kSmemBytes = kBiasOff + BN * 4 + 1024;  // + alignment slack
    // Per-warp epilogue staging of the plain product: two 32-row x 32-column
    // buffers per epilogue warp (sized for fp32) inside the staging area.
    static constexpr uint32_t kWarpBufBytes = 32 * 32 * 4;
    static_assert(8 * kWarpBufBytes <= kEpiBytes, "per-warp staging fits the staging area");
    static_assert(kSmemBytes <= 227 * 1024, "dynamic shared memory of one CTA");
    // Workspace bytes per split piece (both CTAs of a pair).
    static constexpr uint64_t kSlotBytes = static_cast<uint64_t>(CTA_GROUP) * 128 * BN * 4;
    static_assert(kTmemCols <= 512, "TMEM has 512 columns");
    static_assert(AROWS == 128 || AROWS == 64, "A stages hold 128 or 64 rows");
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

// int8 output (the quantising epilogue): v already holds value*scale + zero
// point; round to nearest even (NaN gives 0) and saturate to [-128, 127].
__device__ __forceinline__ int int8_code(float v) { return max(-128, min(127, __float2int_rn(v))); }
template <>
__device__ __forceinline__ float load_out<int8_t>(const int8_t* p) { return static_cast<float>(*p); }
template <>
__device__ __forceinline__ void store_out<int8_t>(int8_t* p, float v) { *p = static_cast<int8_t>(int8_code(v)); }

template <typename OutT>
inline constexpr bool kIsI8 = sizeof(OutT) == 1;

// alpha*acc (+ beta*C) for the 32 columns [col0, col0+32) of one row; `acc`
// holds fp32 bit patterns.  Columns at or beyond N are skipped.
template <typename OutT>
__device__ __forceinline__ void epilogue_store32(OutT* dst, int64_t ldc, int64_t col0, int64_t N,
                                                 const uint32_t (&acc)[32], float alpha, float beta,
                                                 const float (&cold)[32], bool has_beta) {
    if (has_beta) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (col0 + j < N) store_out<OutT>(dst + j * ldc, fmaf(alpha, __uint_as_float(acc[j]), beta * cold[j]));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (col0 + j < N) store_out<OutT>(dst + j * ldc, alpha * __uint_as_float(acc[j]));
        }
    }
}

// The same with the fused epilogue: + bias[column] (the 32 columns' values,
// already in registers so no load waits behind a store), then the activation.
// int8 output: then * qs (this row's scale) + the zero point.
template <typename OutT>
__device__ __forceinline__ void epilogue_store32_fused(OutT* dst, int64_t ldc, int64_t col0, const GemmParams& p,
                                                       const uint32_t (&acc)[32], const float (&cold)[32],
                                                       bool has_beta, const float (&bias)[32], float qs = 1.0f) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        v[j] = (has_beta ? fmaf(p.alpha, __uint_as_float(acc[j]), p.beta * cold[j])
                         : p.alpha * __uint_as_float(acc[j])) + bias[j];
    }
    activation_n(v, p.act);
    if constexpr (kIsI8<OutT>) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaf(v[j], qs, p.qzero);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (col0 + j < p.N) store_out<OutT>(dst + j * ldc, v[j]);
    }
}

// The 32 bias values of columns [col0, col0 + 32), 0 beyond N.
__device__ __forceinline__ void load_bias32(const GemmParams& p, int64_t col0, float (&bias)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) bias[j] = (col0 + j < p.N) ? bias_at(p, col0 + j) : 0.0f;
}

// beta != 0: issue all 32 reads of C before the first write so they are in
// flight together (a write may alias a later read, so the compiler would
// otherwise serialise them).
template <typename OutT>
__device__ __forceinline__ void load_cold32(const OutT* dst, int64_t ldc, int64_t col0, int64_t N,
                                            float (&cold)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) cold[j] = (col0 + j < N) ? load_out<OutT>(dst + j * ldc) : 0.0f;
}

// Swapped product (C^T = B^T A^T): one thread holds 32 consecutive rows of
// one column of C, contiguous in memory.  alpha*acc (+ beta*C) for the first
// `valid` of them, with 16-byte vector accesses when all 32 are in range (the
// run starts 64- or 128-byte aligned: C is 16-byte aligned, ldc*sizeof(T) is a
// multiple of 16 and the run starts at a multiple of 32 rows).
// With FUSED, every value then gets + bias (the one bias value of this row
// of D, a column of C) and the activation before it is stored.  int8 output
// (always FUSED, beta == 0): then * qs32[j] (the scales of these 32 rows of
// C, 16-byte aligned) + zero point, 32 codes in two 16-byte stores.
template <typename OutT, bool FUSED = false>
__device__ __forceinline__ void store_run32(OutT* dst, int64_t valid, const uint32_t (&acc)[32], float alpha,
                                            float beta, bool has_beta, float bias_v = 0.0f, int act = kActNone,
                                            const float* qs32 = nullptr, float zp = 0.0f) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = alpha * __uint_as_float(acc[j]);
    if (valid >= 32) {
        if constexpr (kIsI8<OutT>) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += bias_v;
            activation_n(v, act);
            const float4* s4 = reinterpret_cast<const float4*>(qs32);
            uint32_t w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 sc = __ldg(s4 + q);
                const uint32_t c0 = static_cast<uint8_t>(int8_code(fmaf(v[4 * q], sc.x, zp)));
                const uint32_t c1 = static_cast<uint8_t>(int8_code(fmaf(v[4 * q + 1], sc.y, zp)));
                const uint32_t c2 = static_cast<uint8_t>(int8_code(fmaf(v[4 * q + 2], sc.z, zp)));
                const uint32_t c3 = static_cast<uint8_t>(int8_code(fmaf(v[4 * q + 3], sc.w, zp)));
                w[q] = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else if constexpr (sizeof(OutT) == 4) {
            float4* d4 = reinterpret_cast<float4*>(dst);
            if (has_beta) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 o = d4[q];
                    v[4 * q + 0] = fmaf(alpha, __uint_as_float(acc[4 * q + 0]), beta * o.x);
                    v[4 * q + 1] = fmaf(alpha, __uint_as_float(acc[4 * q + 1]), beta * o.y);
                    v[4 * q + 2] = fmaf(alpha, __uint_as_float(acc[4 * q + 2]), beta * o.z);
                    v[4 * q + 3] = fmaf(alpha, __uint_as_float(acc[4 * q + 3]), beta * o.w);
                }
            }
            if constexpr (FUSED) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += bias_v;
                activation_n(v, act);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            if (has_beta) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 o = d4[q];
                    const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[h]);
                        v[8 * q + 2 * h] = fmaf(alpha, __uint_as_float(acc[8 * q + 2 * h]), beta * __low2float(b2));
                        v[8 * q + 2 * h + 1] =
                            fmaf(alpha, __uint_as_float(acc[8 * q + 2 * h + 1]), beta * __high2float(b2));
                    }
                }
            }
            if constexpr (FUSED) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += bias_v;
                activation_n(v, act);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * q + 2 * h], v[8 * q + 2 * h + 1]);
                    w[h] = *reinterpret_cast<const uint32_t*>(&b2);
                }
                d4[q] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < valid) {
                float x = v[j];
                if (has_beta) x = fmaf(alpha, __uint_as_float(acc[j]), beta * load_out<OutT>(dst + j));
                if constexpr (FUSED) x = activation(x + bias_v, act);
                if constexpr (kIsI8<OutT>) x = fmaf(x, __ldg(qs32 + j), zp);
                store_out<OutT>(dst + j, x);
            }
        }
    }
}

constexpr uint32_t kEpiBarrier = 1;     // named barrier id for the 4 epilogue warps
constexpr uint32_t kEpiThreads = 128;

// tmC maps C (column-major M x N) in 128-row x 32-column boxes for the
// epilogue's TMA loads / stores and L2 prefetches; tmW maps the stream-K
// workspace (fp32, 128 rows x [slot][CTA of pair][BN] columns) the same way.
// SWAP: the launch computes D = C^T (the host swapped A with B and M with N);
// D's rows are C's columns, so the epilogue writes each TMEM row as a
// contiguous run of one column of C (D row-major with leading dimension ldc).
// KS = 2 (transposed product only): a cluster of two CTAs computes each tile,
// CTA 0 over the first half of its k-blocks and CTA 1 over the second half.
// Each CTA then finishes half of the tile's columns: it writes its fp32
// partial of the other half into the peer's epilogue staging area
// ([column][row], through distributed shared memory), adds the partial the
// peer wrote into its own staging area to its accumulator, and stores.  Per
// CTA, xfull (one arrival per epilogue warp of the peer) says the peer's
// partial is in this CTA's staging area, xfree says the peer has read its
// own (so this CTA may write it again).
// NS: MMAs per K step.  NS = 2 issues each K step as two MMAs of width
// BN/2 that share the A operand and write the two column halves of the
// accumulator.  It doubles the MMA instructions; measured on GB300 one MMA
// per K step already runs at the full rate of 8192 FLOP per clock per SM
// when the K step holds at least about 116 clocks of work, so NS = 2 is an
// option that measured slower.  For a CTA pair the halves of the tile that each MMA
// reads must sit at the same shared-memory offset in both CTAs, so each CTA
// loads its B rows as NS boxes: box h holds tile columns
// [h*BN/NS + rank*BN/(2*NS), ...), and the accumulator columns stay in tile
// order.
template <int CTA_GROUP, int BN, int STAGES, int AROWS, bool SWAP, typename OutT, int IN = 0, int KS = 1, int NS = 1>
__global__ void __launch_bounds__(192, 1)
    gemm_bf16_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW,
                        const GemmParams p) {
    using Cfg = GemmCfg<CTA_GROUP, BN, STAGES, AROWS, IN, KS>;
    static_assert(NS == 1 || (NS == 2 && (!SWAP || CTA_GROUP == 1) && (Cfg::kRowsB / 2) % 8 == 0 &&
                              (BN / 2) % 16 == 0),
                  "split MMAs: whole swizzle atoms of B per half, MMA widths a multiple of 16");
    constexpr int kRowsBh = Cfg::kRowsB / NS;  // B rows of one split MMA in this CTA
    static_assert(!SWAP || CTA_GROUP == 1 || (KS == 1 && AROWS == 64), "pairs run the swapped product with "
                  "64-row A stages and no K split");
    static_assert(AROWS == 128 || SWAP || CTA_GROUP == 1, "half-height A tiles: single CTAs or the swapped pairs");
    static_assert(KS == 1 || (KS == 2 && SWAP && BN % 64 == 0 && Cfg::kEpiBytes >= 128u * (BN / 2) * 4u),
                  "the K split exchanges half an fp32 tile through the staging area");
    constexpr int kCluster = CTA_GROUP * KS;
    // Transposed product on a CTA pair: each CTA loads rows_a (<= 64) rows of
    // the MMA's A operand into a 64-row stage; the pair's M = 256 MMA reads
    // 128 rows per CTA, the rows past rows_a (stale rows, or the next stage)
    // give accumulator rows that are never stored.  A pair tile is 2*rows_a
    // rows of D, so the tiles can be sized to give every SM one.
    constexpr bool kPairSwap = SWAP && CTA_GROUP == 2;
    const int rows_a = kPairSwap ? p.rows_a : Cfg::kRowsA;
    const int tile_m = kPairSwap ? 2 * p.rows_a : Cfg::kBM;
    extern __shared__ uint8_t smem_raw[];

    // 1 KB-aligned carve-up: [A stages][B stages][barriers][tmem slot][abort][last flag]
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
    // C chunk loads of epilogue warp q (0..3) into its buffer b.
    auto cold_bar = [&](uint32_t q, uint32_t b) { return bar0 + 8u * (2 * STAGES + 5 + 2 * q + b); };
    const uint32_t xfull_bar = bar0 + 8u * (2 * STAGES + 13);  // KS = 2: the peer's partial is in this CTA's area
    const uint32_t xfree_bar = bar0 + 8u * (2 * STAGES + 14);  // KS = 2: the peer has read its own area
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kBarOff + Cfg::kNumBars * 8);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    volatile uint32_t* never_flag = tmem_slot + 2;  // stays 0: drains wait for copies even after an abort

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t crank = (kCluster > 1) ? cluster_ctarank() : 0u;
    const uint32_t rank = (CTA_GROUP == 2) ? crank : 0u;  // position in the MMA pair
    const uint32_t ks_rank = (KS == 2) ? crank : 0u;       // which half of each tile's k-blocks
    // This CTA's share of a unit's k-blocks: the first half (rounded up) for
    // CTA 0 of a K-split cluster, the rest for CTA 1.
    auto ks_range = [&](WorkUnit& u) {
        if constexpr (KS == 2) {
            const int mid = u.kb0 + (u.kb1 - u.kb0 + 1) / 2;
            if (ks_rank == 0) u.kb1 = mid;
            else u.kb0 = mid;
        }
    };
    const int cluster_id = blockIdx.x / kCluster;
    const int num_clusters = gridDim.x / kCluster;
    auto tile_of = [&](int unit_tile, int& tm, int& tn) { unit_tile_of(p, unit_tile, tm, tn); };

    // Single-CTA MMAs: the producer needs nothing but its own barriers, so it
    // starts loading as soon as they are initialised, while the TMEM
    // allocation and the (cluster) barrier complete for the other warps.
    constexpr bool kEarlyProducer = CTA_GROUP == 1;
    if (threadIdx.x == 0) {
        // The descriptors' first fetch overlaps the set-up.
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 2 && lane == 0) tma_prefetch_desc(&tmC);
    // The producer's first unit.  Its parameter reads are the first of the
    // launch and come from memory (about a microsecond): a single-CTA
    // producer works it out before the set-up; a CTA pair's producer between
    // arriving at the cluster barrier and waiting on it, so that the two
    // latencies overlap.
    UnitIter pit(cluster_id, num_clusters);
    WorkUnit pu{};
    bool p_have = false;
    int p_tm = 0, p_tn = 0;
    auto first_unit = [&]() {
        pit.start(p);
        p_have = pit.next(p, pu);
        if (p_have) {
            ks_range(pu);
            tile_of(pu.tile, p_tm, p_tn);
        }
    };
    if (kEarlyProducer && warp == 0 && lane == 0) first_unit();
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
        for (uint32_t c = 0; c < 8; ++c) mbar_init(cold_bar(c >> 1, c & 1u), 1);
        mbar_init(xfull_bar, 4);
        mbar_init(xfree_bar, 4);
        *abort_flag = 0u;
        *never_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc<CTA_GROUP>(smem_u32(tmem_slot), Cfg::kTmemAlloc);
    if (kEarlyProducer && warp == 0) {
        // Arrive now, wait (cluster) after the loads are issued.
        __syncwarp();
        if constexpr (kCluster == 1) {
            named_barrier_arrive(0, Cfg::kThreads);
        } else {
            cluster_arrive();
        }
    } else {
        tc_fence_before_sync();
        if constexpr (kCluster == 1) {
            if constexpr (kEarlyProducer) {
                named_barrier_sync(0, Cfg::kThreads);
            } else {
                __syncthreads();
            }
        } else {
            cluster_arrive();
            if (!kEarlyProducer && warp == 0 && lane == 0) first_unit();
            __syncwarp();
            cluster_wait();
        }
        tc_fence_after_sync();
    }
    const uint32_t tmem_base = *tmem_slot;  // not read by an early producer
    const WaitCtx wctx{abort_flag, p.timeout_ns};
    // Drains wait for this CTA's own copies and MMAs to finish whether or not
    // another role gave up (bounded by the same limit): the CTA may not exit,
    // nor free its TMEM, while a TMA copy or an MMA still uses them.
    const WaitCtx dctx{never_flag, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint64_t issued = 0;
            bool ok = true;
            // Launched as a programmatic dependent of the previous kernel on
            // the stream, the set-up above may have overlapped its tail; no
            // global memory is read before that kernel has completed.
            grid_dependency_wait();
            while (ok && p_have) {
                const WorkUnit u = pu;
                const int tm = p_tm, tn = p_tn;
                const int a_row = tm * tile_m + static_cast<int>(rank) * rows_a;
                const CUtensorMap* mB = &tmB;
                const uint32_t stage_tx = kPairSwap ? CTA_GROUP * (static_cast<uint32_t>(rows_a) * 128u + Cfg::kBBytes)
                                                    : Cfg::kStageTx;
                // One operand tile: K-major, one box of 64 K values by `rows`
                // rows; MN-major, boxes of 64 MN values by 64 K rows, 8 KB
                // apart.  Same bytes either way.
                auto load_tile = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int kb, int row0, int rows,
                                     bool mn) {
                    if (!mn) {
                        if constexpr (CTA_GROUP == 1) tma_load_2d(dst, map, bar, kb * Cfg::kBK, row0);
                        else tma_load_2d_pair(dst, map, bar, kb * Cfg::kBK, row0);
                    } else {
                        for (int t = 0; t < rows; t += 64) {
                            if constexpr (CTA_GROUP == 1) tma_load_2d(dst + t * 128, map, bar, row0 + t, kb * 64);
                            else tma_load_2d_pair(dst + t * 128, map, bar, row0 + t, kb * 64);
                        }
                    }
                };
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!wait_phase<false>(empty_bar(stage), phase ^ 1u, wctx, kWhereProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sA0 + stage * Cfg::kABytes;
                    const uint32_t sb = sB0 + stage * Cfg::kBBytes;
                    if (p.withhold_kb >= 0 && blockIdx.x == 0 && issued == static_cast<uint64_t>(p.withhold_kb)) {
                        // Self test: this stage's phase is never completed.
                    } else if constexpr (CTA_GROUP == 1) {
                        mbar_arrive_expect_tx(full_bar(stage), stage_tx);
                        load_tile(sa, &tmA, full_bar(stage), kb, a_row, Cfg::kRowsA, p.a_mn != 0);
                        load_tile(sb, mB, full_bar(stage), kb, tn * BN, Cfg::kRowsB, p.b_mn != 0);
                    } else {
                        // Both CTAs' bytes land on the leader's barrier.
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), stage_tx);
                        const uint32_t fb = map_to_cta(full_bar(stage), 0);
                        load_tile(sa, &tmA, fb, kb, a_row, Cfg::kRowsA, p.a_mn != 0);
#pragma unroll
                        for (int h = 0; h < NS; ++h)
                            load_tile(sb + h * kRowsBh * 128, mB, fb, kb,
                                      tn * BN + h * (BN / NS) + static_cast<int>(rank) * kRowsBh, kRowsBh,
                                      p.b_mn != 0);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                // The next unit, worked out while this one's loads are in flight.
                p_have = pit.next(p, pu);
                if (p_have) {
                    ks_range(pu);
                    tile_of(pu.tile, p_tm, p_tn);
                }
            }
            // Every load is issued: a dependent kernel (the stream-K
            // reduction) may begin launching; it waits for this grid to
            // complete before it reads anything.
            grid_launch_dependents();
            // Drain: every load this thread issued has landed before the CTA
            // may exit.  The leader (or a lone CTA) sees that on its full
            // barriers; a pair's second CTA sees it when the leader's MMA
            // frees the stage again.
            for (int s = 0; s < STAGES; ++s) {
                if (issued <= static_cast<uint64_t>(s)) break;
                const uint64_t times = (issued - s - 1) / STAGES + 1;
                const uint32_t par = static_cast<uint32_t>((times - 1) & 1u);
                if (CTA_GROUP == 1 || rank == 0) {
                    wait_phase<false>(full_bar(s), par, dctx, kWhereDrain);
                } else {
                    wait_phase<false>(empty_bar(s), par, dctx, kWhereDrain);
                }
            }
        }
        if constexpr (kEarlyProducer && kCluster > 1) {
            // The wait that goes with the early arrive above.
            __syncwarp();
            cluster_wait();
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0 && (CTA_GROUP == 1 || rank == 0)) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            // The units' MMAs.  MN: either operand MN-major (descriptors and
            // steps chosen per operand at run time); otherwise the K-major
            // code with constant steps.  The single thread issuing MMAs is on
            // the critical path, so the common layout keeps its own copy.
            auto issue_units = [&](auto mn_tag) {
            constexpr bool MN = decltype(mn_tag)::value;
            // Bits 15 / 16 of the instruction descriptor: A / B MN-major.
            const uint32_t kIdesc = (IN == 1 ? idesc_f8_f32(Cfg::kBM, BN / NS, static_cast<uint32_t>(p.in_fmt) & 1u,
                                                            (static_cast<uint32_t>(p.in_fmt) >> 1) & 1u)
                                             : idesc_bf16_f32(Cfg::kBM, BN / NS)) |
                                    (MN && p.a_mn ? (1u << 15) : 0u) | (MN && p.b_mn ? (1u << 16) : 0u);
            // Descriptor step per MMA: 32 bytes along a K-major row, two
            // 1 KB K groups in an MN-major tile (in 16-byte units).
            const uint32_t a_step = MN && p.a_mn ? 128u : 2u, b_step = MN && p.b_mn ? 128u : 2u;
            bool ok = true;
            UnitIter it(cluster_id, num_clusters);
            it.start(p);
            WorkUnit u;
            while (ok && it.next(p, u)) {
                ks_range(u);
                if (!wait_phase<CTA_GROUP == 2>(tempty_bar(acc), acc_phase ^ 1u, wctx, kWhereMma)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                const uint32_t idesc = kIdesc;
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!wait_phase<false>(full_bar(stage), phase, wctx, kWhereMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = sA0 + stage * Cfg::kABytes, sb = sB0 + stage * Cfg::kBBytes;
                    const uint64_t ad = MN && p.a_mn ? sdesc_mnmajor_sw128(sa) : sdesc_kmajor_sw128(sa);
                    const uint64_t bd = MN && p.b_mn ? sdesc_mnmajor_sw128(sb) : sdesc_kmajor_sw128(sb);
#pragma unroll
                    for (int k = 0; k < Cfg::kBK / Cfg::kUmmaK; ++k) {
#pragma unroll
                        for (int h = 0; h < NS; ++h) {
                            // Split MMA h: its B rows start kRowsBh rows (whole
                            // 1 KB swizzle atoms, or 8 KB MN-major boxes of 64
                            // rows) further on; it writes columns h*BN/NS.. .
                            const uint32_t bh = static_cast<uint32_t>(h) * kRowsBh * 8u;
                            const uint32_t dh = d_tmem + static_cast<uint32_t>(h) * (BN / NS);
                            if constexpr (MN) {
                                mma_tc<CTA_GROUP, IN>(dh, ad + a_step * k, bd + bh + b_step * k, idesc,
                                                      (kb != u.kb0 || k != 0) ? 1u : 0u);
                            } else {
                                // +32 bytes along K per step: (32 >> 4) = 2 in the address field.
                                mma_tc<CTA_GROUP, IN>(dh, ad + 2u * k, bd + bh + 2u * k, idesc,
                                                      (kb != u.kb0 || k != 0) ? 1u : 0u);
                            }
                        }
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
            };
            if (p.a_mn || p.b_mn) {
                issue_units(std::true_type{});
            } else {
                issue_units(std::false_type{});
            }

            // Drain: all MMAs issued by this thread have completed.
            if constexpr (CTA_GROUP == 1) {
                mma_commit(drain_bar);
            } else {
                mma_commit_pair(drain_bar, 0x1);
            }
            wait_phase<false>(drain_bar, 0, dctx, kWhereDrain);
        }
    } else {
        // --------------------------------------------------- epilogue --
        // Warp w may only touch TMEM lanes 32*(w%4) .. 32*(w%4)+31.
        const uint32_t q = warp & 3u;
        const uint32_t row_local = q * 32u + lane;  // 0..127 within this CTA's rows
        OutT* C = static_cast<OutT*>(p.C);
        const bool has_beta = p.beta != 0.0f;
        const bool fused = kIsI8<OutT> || has_epilogue(p);  // int8 output always takes the fused path
        float* bias_s = reinterpret_cast<float*>(smem + Cfg::kBiasOff);
        // Stream-K pieces: two staging buffers shared by the four epilogue
        // warps, each one 128-row x 32-column fp32 chunk with rows fastest
        // (the layout of the TMA box); one thread (warp 2, lane 0) issues
        // their TMA stores.  Whole tiles use per-warp buffers (below).
        const bool leader = (warp == 2 && lane == 0);
        uint32_t nchunk = 0;      // stream-K chunks staged so far; chunk i uses buffer i & 1
        uint32_t cold_phase = 0;  // bit b: parity of the next completion of this warp's cold_bar(q, b)
        bool aborted = false;
        uint32_t acc = 0, acc_phase = 0;
        uint32_t xph = 0;  // KS = 2: parity of the next exchange
        grid_dependency_wait();  // as the producer: after the previous kernel on the stream
        UnitIter it(cluster_id, num_clusters);
        it.start(p);
        WorkUnit u;
        while (!aborted && it.next(p, u)) {
            int tm, tn;
            tile_of(u.tile, tm, tn);
            const int row_blk = tm * tile_m + static_cast<int>(rank) * (kPairSwap ? rows_a : 128);  // this CTA's rows
            const int64_t colt = static_cast<int64_t>(tn) * BN;  // first column of the tile
            const int ncols = BN;
            // beta*C: each warp starts pulling its rows of the C tile into L2
            // now; the tile's mainloop hides the memory latency.
            const int wrow = row_blk + 32 * static_cast<int>(q);  // this warp's first row (plain product)
            if (!SWAP && has_beta && lane == 0 && wrow < p.M) {
                for (int c = 0; c < ncols && colt + c < p.N; c += 32)
                    tma_prefetch_l2_2d(&tmC, wrow, static_cast<int32_t>(colt + c));
            }
            // The staging area is reused by this unit: every store of earlier
            // units has finished reading it (the barrier below publishes that).
            if (lane == 0) tma_store_wait_read<0>();
            const int64_t row = static_cast<int64_t>(row_blk) + row_local;
            const bool row_ok = row < p.M && (!kPairSwap || static_cast<int>(row_local) < rows_a);
            // Fused epilogue: fetch the tile's bias now, while the mainloop
            // runs.  Plain product: the tile's BN column values go to shared
            // memory (every reader of the previous tile's values has passed
            // the barrier that ends that tile); transposed product: this
            // thread's row has one value.
            float bias_v = 0.0f;
            float qs = 1.0f;  // int8 output: this row's scale (plain product)
            if constexpr (kIsI8<OutT> && !SWAP) {
                if (row_ok) qs = __ldg(p.qscale + row);
            }
            if (fused && u.slot < 0) {
                if constexpr (SWAP) {
                    if (row_ok) bias_v = bias_at(p, row);
                } else {
                    for (int c = static_cast<int>(row_local); c < BN; c += 128)
                        bias_s[c] = (colt + c < p.N) ? bias_at(p, colt + c) : 0.0f;
                }
            }
            uint32_t ok = 1;
            if (lane == 0) ok = wait_phase<false>(tfull_bar(acc), acc_phase, wctx, kWhereEpilogue) ? 1u : 0u;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            // All four epilogue warps agree before going on, so none is left
            // alone at a named barrier below if another one gave up.
            if (!named_barrier_and(kEpiBarrier, kEpiThreads, ok != 0u)) break;
            tc_fence_after_sync();
            const uint32_t tbase = tmem_base + ((q * 32u) << 16) + acc * BN;

            if (KS == 2) {
                // K-split tile: each CTA finishes half of the tile's columns
                // (D columns = rows of C).  It writes the fp32 partial of the
                // other half into its peer's staging area (distributed
                // shared memory: posted stores, one contiguous 128-byte run
                // per warp and column), then adds the partial its peer wrote
                // into its own staging area to its accumulator and stores.
                // Two partials, so the sum does not depend on which CTA adds
                // it up.  xfree: the peer has read its staging area (this
                // CTA may write it again); xfull: the peer's partial is in
                // this CTA's staging area.
                const uint32_t peer = ks_rank ^ 1u;
                const int half = ncols / 2;
                const int mine = static_cast<int>(ks_rank) * half, theirs = static_cast<int>(peer) * half;
                uint32_t okx = 1;
                if (lane == 0) okx = wait_phase<true>(xfree_bar, xph ^ 1u, wctx, kWhereEpilogue) ? 1u : 0u;
                okx = __shfl_sync(0xffffffffu, okx, 0);
                if (!named_barrier_and(kEpiBarrier, kEpiThreads, okx != 0u)) break;
                const float* xb = reinterpret_cast<const float*>(smem + Cfg::kEpiOff) + row_local;
                const uint32_t xpeer = map_to_cta(base + Cfg::kEpiOff, peer) + row_local * 4u;
#pragma unroll 1
                for (int c = 0; c < half; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tbase + theirs + c, r);
                    tmem_ld_wait32(r);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        st_dsmem_f32(xpeer + static_cast<uint32_t>(c + j) * 512u, __uint_as_float(r[j]));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(map_to_cta(xfull_bar, peer));
                okx = 1;
                if (lane == 0) okx = wait_phase<true>(xfull_bar, xph, wctx, kWhereEpilogue) ? 1u : 0u;
                okx = __shfl_sync(0xffffffffu, okx, 0);
                if (!named_barrier_and(kEpiBarrier, kEpiThreads, okx != 0u)) break;
#pragma unroll 1
                for (int c = 0; c < half; c += 32) {
                    const int64_t col0 = colt + mine + c;
                    if (col0 >= p.N) break;
                    uint32_t r[32];
                    tmem_ld32(tbase + mine + c, r);
                    float x[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = xb[(c + j) * 128];
                    tmem_ld_wait32(r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + x[j]);
                    if (row_ok) {
                        OutT* dst = C + row * p.ldc + col0;
                        if (fused) {
                            store_run32<OutT, true>(dst, p.N - col0, r, p.alpha, p.beta, has_beta, bias_v, p.act,
                                                    p.qscale + col0, p.qzero);
                        } else {
                            store_run32<OutT>(dst, p.N - col0, r, p.alpha, p.beta, has_beta);
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(tempty_bar(acc));
                    mbar_arrive_cluster(map_to_cta(xfree_bar, peer));
                }
                xph ^= 1u;
            } else if (SWAP && u.slot < 0) {
                // D row `row` = column `row` of C; D columns = rows of C.
#pragma unroll 1
                for (int c = 0; c < ncols; c += 32) {
                    const int64_t col0 = colt + c;
                    if (col0 >= p.N) break;
                    uint32_t r[32];
                    tmem_ld32(tbase + c, r);
                    tmem_ld_wait32(r);
                    if (row_ok) {
                        OutT* dst = C + row * p.ldc + col0;
                        if (fused) {
                            store_run32<OutT, true>(dst, p.N - col0, r, p.alpha, p.beta, has_beta, bias_v, p.act,
                                                    p.qscale + col0, p.qzero);
                        } else {
                            store_run32<OutT>(dst, p.N - col0, r, p.alpha, p.beta, has_beta);
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
            } else if (u.slot < 0) {
                // Whole tile, chunk by chunk, each epilogue warp on its own 32
                // rows: (TMA load of its rows of C ->) TMEM -> alpha*acc
                // (+ beta*C) in the warp's staging buffer -> TMA store of its
                // 32-row x 32-column box (the store clips columns >= N and
                // rows >= M).  The warps do not wait for one another: lane 0
                // of each warp issues, and waits for, its own copies.  The
                // next chunk's TMEM load is issued before this chunk is
                // converted.  A warp whose rows end inside a 16-byte granule
                // at row M stores with masked plain stores instead (the TMA
                // store would also write rows M.. of the ldc padding).
                const int64_t width = (p.N - colt) < ncols ? (p.N - colt) : ncols;
                const int nch = static_cast<int>((width + 31) / 32);
                const bool w_rows = wrow < p.M;
                const bool w_tma = wrow + 32 <= p.M || ((static_cast<int64_t>(p.M) * sizeof(OutT)) % 16) == 0;
                const uint32_t wbuf = base + Cfg::kEpiOff + q * 2u * Cfg::kWarpBufBytes;
                OutT* wsp0 = reinterpret_cast<OutT*>(smem + Cfg::kEpiOff + q * 2u * Cfg::kWarpBufBytes);
                constexpr uint32_t kWarpBufElems = Cfg::kWarpBufBytes / sizeof(OutT);
                constexpr uint32_t kWarpChunkBytes = 32 * 32 * sizeof(OutT);
                bool wok = true;
                if (w_rows && !w_tma) {
#pragma unroll 1
                    for (int c = 0; c < ncols; c += 32) {
                        const int64_t col0 = colt + c;
                        if (col0 >= p.N) break;
                        OutT* dst = C + col0 * p.ldc + row;
                        float cold[32];
                        if (has_beta && row_ok) load_cold32<OutT>(dst, p.ldc, col0, p.N, cold);
                        uint32_t r[32];
                        tmem_ld32(tbase + c, r);
                        tmem_ld_wait32(r);
                        if (row_ok) {
                            if (fused) {
                                float bj[32];
#pragma unroll
                                for (int j = 0; j < 32; ++j) bj[j] = bias_s[c + j];
                                epilogue_store32_fused<OutT>(dst, p.ldc, col0, p, r, cold, has_beta, bj, qs);
                            } else {
                                epilogue_store32<OutT>(dst, p.ldc, col0, p.N, r, p.alpha, p.beta, cold, has_beta);
                            }
                        }
                    }
                } else if (w_rows) {
                    const bool load_c = has_beta;
                    if (load_c && lane == 0) {
                        mbar_arrive_expect_tx(cold_bar(q, 0), kWarpChunkBytes);
                        tma_load_2d(wbuf, &tmC, cold_bar(q, 0), wrow, static_cast<int32_t>(colt));
                    }
                    uint32_t rn[32];
                    tmem_ld32(tbase, rn);
#pragma unroll 1
                    for (int i = 0; i < nch; ++i) {
                        const int64_t col0 = colt + 32 * i;
                        const uint32_t b = static_cast<uint32_t>(i) & 1u;
                        OutT* sp = wsp0 + b * kWarpBufElems;
                        uint32_t r[32];
                        tmem_ld_wait32(rn);
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = rn[j];
                        if (i + 1 < nch) tmem_ld32(tbase + 32 * (i + 1), rn);
                        if (load_c) {
                            if (lane == 0 && i + 1 < nch) {
                                // The other buffer's last store (chunk i - 1)
                                // must be done reading it.
                                tma_store_wait_read<0>();
                                mbar_arrive_expect_tx(cold_bar(q, b ^ 1u), kWarpChunkBytes);
                                tma_load_2d(wbuf + (b ^ 1u) * Cfg::kWarpBufBytes, &tmC, cold_bar(q, b ^ 1u), wrow,
                                            static_cast<int32_t>(col0 + 32));
                            }
                            uint32_t okc = 1;
                            if (lane == 0) okc = wait_phase<false>(cold_bar(q, b), (cold_phase >> b) & 1u, wctx,
                                                                   kWhereEpilogue) ? 1u : 0u;
                            okc = __shfl_sync(0xffffffffu, okc, 0);
                            cold_phase ^= 1u << b;
                            if (okc == 0u) {
                                wok = false;
                                if (i + 1 < nch) {
                                    tmem_ld_wait32(rn);
                                    // The next chunk's load of C is in flight:
                                    // it lands before the CTA moves on.
                                    if (lane == 0)
                                        (void)wait_phase<false>(cold_bar(q, b ^ 1u), (cold_phase >> (b ^ 1u)) & 1u,
                                                                dctx, kWhereDrain);
                                    __syncwarp();
                                }
                                break;
                            }
                        } else {
                            // This buffer's previous store (two chunks ago)
                            // must be done reading it.
                            if (lane == 0 && i >= 2) tma_store_wait_read<1>();
                            __syncwarp();
                        }
                        if (fused) {
                            // + bias[column] (staged; 0 beyond N, where the
                            // store clips anyway), activation.
                            float bj[32];
                            const float4* b4 = reinterpret_cast<const float4*>(bias_s + 32 * i);
#pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                const float4 t4 = b4[t];
                                bj[4 * t] = t4.x;
                                bj[4 * t + 1] = t4.y;
                                bj[4 * t + 2] = t4.z;
                                bj[4 * t + 3] = t4.w;
                            }
                            float vv[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                float v = p.alpha * __uint_as_float(r[j]);
                                if (load_c) v = fmaf(p.alpha, __uint_as_float(r[j]), p.beta * load_out<OutT>(sp + j * 32 + lane));
                                vv[j] = v + bj[j];
                            }
                            activation_n(vv, p.act);
                            if constexpr (kIsI8<OutT>) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) vv[j] = fmaf(vv[j], qs, p.qzero);
                            }
#pragma unroll
                            for (int j = 0; j < 32; ++j) store_out<OutT>(sp + j * 32 + lane, vv[j]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                OutT* e = sp + j * 32 + lane;
                                float v = p.alpha * __uint_as_float(r[j]);
                                if (load_c) v = fmaf(p.alpha, __uint_as_float(r[j]), p.beta * load_out<OutT>(e));
                                store_out<OutT>(e, v);
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmC, wbuf + b * Cfg::kWarpBufBytes, wrow, static_cast<int32_t>(col0));
                            tma_store_commit();
                        }
                    }
                }
                // Every warp is done with the tile (or one gave up).
                if (!named_barrier_and(kEpiBarrier, kEpiThreads, wok)) {
                    aborted = true;
                    break;
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
            } else {
                // Stream-K piece: stage the fp32 partial tile (all 128 rows,
                // all BN columns) and TMA-store it to this piece's slot.
                float* fsp0 = reinterpret_cast<float*>(smem + Cfg::kEpiOff);
                constexpr uint32_t kFBufElems = Cfg::kEpiBufBytes / 4;
                const int ws_col0 = (u.slot * CTA_GROUP + static_cast<int>(rank)) * BN;
#pragma unroll 1
                for (int i = 0; i < BN / 32; ++i) {
                    const uint32_t b = nchunk & 1u;
                    float* sp = fsp0 + b * kFBufElems;
                    uint32_t r[32];
                    tmem_ld32(tbase + 32 * i, r);
                    if (leader && nchunk >= 2) tma_store_wait_read<1>();
                    named_barrier_sync(kEpiBarrier, kEpiThreads);
                    tmem_ld_wait32(r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) sp[j * 128 + row_local] = __uint_as_float(r[j]);
                    fence_proxy_async_smem();
                    named_barrier_sync(kEpiBarrier, kEpiThreads);
                    if (leader) {
                        tma_store_2d(&tmW, base + Cfg::kEpiOff + b * Cfg::kEpiBufBytes, 0, ws_col0 + 32 * i);
                        tma_store_commit();
                    }
                    ++nchunk;
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
            }
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        // Every TMA store has completed before the CTA exits.
        if (lane == 0) tma_store_wait_all();
        __syncwarp();
    }

    // ------------------------------------------------------- teardown --
    grid_launch_dependents();
    __syncwarp();
    tc_fence_before_sync();
    if constexpr (kCluster == 1) {
        __syncthreads();
    } else {
        cluster_sync();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CTA_GROUP>(tmem_base, Cfg::kTmemAlloc);
    }
}

// Stream-K reduction: one block per (shared tile, CTA of pair, 32-column
// chunk), one thread per row.  Adds the tile's pieces in K order (the same
// order whatever order they were computed in), then alpha/beta, the output
// cast and masked, coalesced stores (a warp writes 32 consecutive rows of a
// column).  Partials: fp32, 128 rows x [slot][CTA of pair][BN] columns.
// Launched as a programmatic dependent of the GEMM, so that its launch
// overlaps the GEMM's last units; it waits for the whole GEMM grid, and for
// its memory operations, before it reads a partial.
constexpr int kSkReduceCols = 32;   // columns per reduction block

template <int CTA_GROUP, int BN>
__host__ __device__ constexpr int sk_reduce_blocks_per_tile() { return CTA_GROUP * (BN / kSkReduceCols); }

template <int CTA_GROUP, int BN, bool SWAP, typename OutT>
__global__ void __launch_bounds__(128)
    sk_reduce_kernel(const float* __restrict__ ws, const GemmParams p, int num_clusters) {
    static_assert(BN % kSkReduceCols == 0, "tile width must be a whole number of reduction chunks");
    const int chunks = BN / kSkReduceCols;
    const int blk = blockIdx.x;
    const int c = blk % chunks;
    const int rank = (blk / chunks) % CTA_GROUP;
    const int t = blk / (chunks * CTA_GROUP);
    if (t >= p.sk_tiles) return;
    const int row_local = threadIdx.x;
    int tm, tn;
    unit_tile_of(p, p.tiles_dp + t, tm, tn);
    const int64_t row = static_cast<int64_t>(tm) * (128 * CTA_GROUP) + rank * 128 + row_local;
    const int64_t col0 = static_cast<int64_t>(tn) * BN + kSkReduceCols * c;
    // The bias is an input, not written by the GEMM: fetch it before waiting.
    const bool fused = kIsI8<OutT> || has_epilogue(p);
    float bj[32];
    if (fused) {
        if constexpr (SWAP) {
            const float b = row < p.M ? bias_at(p, row) : 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) bj[j] = b;
        } else {
            load_bias32(p, col0, bj);
        }
    }
    grid_dependency_wait();
    if (col0 >= p.N) return;
    const int64_t t_begin = static_cast<int64_t>(t) * p.num_kb;
    const int first = sk_owner(t_begin, p.sk_iters, num_clusters);
    const int last = sk_owner(t_begin + p.num_kb - 1, p.sk_iters, num_clusters);
    const int64_t piece_stride = static_cast<int64_t>(BN) * 128;
    const int64_t base = static_cast<int64_t>(rank * BN + kSkReduceCols * c) * 128 + row_local;
    float sum[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) sum[j] = 0.0f;
    // Two pieces' loads in flight at a time; the additions stay in K order.
    int cl = first;
    for (; cl + 1 <= last; cl += 2) {
        const float* s0 = ws + sk_slot(cl, t_begin, p.sk_iters, num_clusters) * CTA_GROUP * piece_stride + base;
        const float* s1 = ws + sk_slot(cl + 1, t_begin, p.sk_iters, num_clusters) * CTA_GROUP * piece_stride + base;
        float v0[32], v1[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v0[j] = __ldcg(s0 + j * 128);
#pragma unroll
        for (int j = 0; j < 32; ++j) v1[j] = __ldcg(s1 + j * 128);
#pragma unroll
        for (int j = 0; j < 32; ++j) sum[j] = (sum[j] + v0[j]) + v1[j];
    }
    if (cl <= last) {
        const float* s0 = ws + sk_slot(cl, t_begin, p.sk_iters, num_clusters) * CTA_GROUP * piece_stride + base;
#pragma unroll
        for (int j = 0; j < 32; ++j) sum[j] += __ldcg(s0 + j * 128);
    }
    if (row >= p.M) return;
    const bool has_beta = p.beta != 0.0f;
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(sum[j]);
    if constexpr (SWAP) {
        OutT* dst = static_cast<OutT*>(p.C) + row * p.ldc + col0;
        if (fused) {
            store_run32<OutT, true>(dst, p.N - col0, r, p.alpha, p.beta, has_beta, bj[0], p.act, p.qscale + col0,
                                    p.qzero);
        } else {
            store_run32<OutT>(dst, p.N - col0, r, p.alpha, p.beta, has_beta);
        }
    } else {
        OutT* dst = static_cast<OutT*>(p.C) + col0 * p.ldc + row;
        float cold[32];
        if (has_beta) load_cold32<OutT>(dst, p.ldc, col0, p.N, cold);
        if (fused) {
            const float qs = kIsI8<OutT> ? __ldg(p.qscale + row) : 1.0f;
            epilogue_store32_fused<OutT>(dst, p.ldc, col0, p, r, cold, has_beta, bj, qs);
        } else {
            epilogue_store32<OutT>(dst, p.ldc, col0, p.N, r, p.alpha, p.beta, cold, has_beta);
        }
    }
}

// C = beta * C (or 0 when beta == 0): the K == 0 case, where the product is
// an empty sum; with the fused epilogue, act(beta * C + bias[j]).  Only
// p.M, p.N, p.ldc, p.C, p.beta and the epilogue fields are used.
template <typename OutT>
__global__ void scale_c_kernel(const GemmParams p) {
    const int64_t M = p.M, N = p.N;
    const int64_t total = M * N;
    OutT* C = static_cast<OutT*>(p.C);
    const bool fused = has_epilogue(p);
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = idx / M, i = idx - j * M;
        OutT* dst = C + j * p.ldc + i;
        float v = p.beta == 0.0f ? 0.0f : p.beta * load_out<OutT>(dst);
        if (fused) v = activation(v + bias_at(p, j), p.act);
        if constexpr (kIsI8<OutT>) v = fmaf(v, __ldg(p.qscale + i), p.qzero);
        store_out<OutT>(dst, v);
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
