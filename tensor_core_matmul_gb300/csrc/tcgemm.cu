// Host side of the tcgemm C ABI: argument checks, TMA descriptor encoding,
// variant choice and kernel launch.  See include/tcgemm.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "../../include/tcgemm.h"
#include "gemm_kernel.cuh"

namespace {

thread_local char t_last_error[512];

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
}

std::atomic<uint64_t> g_launches{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<EncodeTiledFn>(p);
        }
    });
    return fn;
}

// cuTensorMapEncodeTiled with a small per-thread memo: repeated calls on the
// same buffers and shapes (the common case in a loop) reuse the descriptor
// instead of encoding it again.  A descriptor depends only on the arguments
// below, so a hit is always the descriptor the driver would return.
struct MapKey {
    CUtensorMapDataType dt;
    const void* ptr;
    cuuint64_t dims[2];
    cuuint64_t stride;
    cuuint32_t box[2];
    CUtensorMapSwizzle swizzle;
    CUtensorMapL2promotion promo;
    bool operator==(const MapKey& o) const {
        return dt == o.dt && ptr == o.ptr && dims[0] == o.dims[0] && dims[1] == o.dims[1] && stride == o.stride &&
               box[0] == o.box[0] && box[1] == o.box[1] && swizzle == o.swizzle && promo == o.promo;
    }
};

CUresult encode_2d(CUtensorMap* m, const MapKey& k) {
    constexpr int kMemo = 16;
    thread_local MapKey keys[kMemo];
    thread_local CUtensorMap maps[kMemo];
    thread_local bool used[kMemo] = {};
    thread_local int next = 0;
    for (int i = 0; i < kMemo; ++i) {
        if (used[i] && keys[i] == k) {
            *m = maps[i];
            return CUDA_SUCCESS;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t strides[1] = {k.stride};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(m, k.dt, 2, const_cast<void*>(k.ptr), k.dims, strides, k.box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, k.swizzle, k.promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
        keys[next] = k;
        maps[next] = *m;
        used[next] = true;
        next = (next + 1) % kMemo;
    }
    return r;
}

uint64_t timeout_ns() {
    static uint64_t ns = [] {
        const char* s = std::getenv("TCGEMM_TIMEOUT_MS");
        double ms = s ? std::atof(s) : 0.0;
        if (!(ms > 0.0)) ms = 2000.0;
        return static_cast<uint64_t>(ms * 1e6);
    }();
    return ns;
}

// ------------------------------------------------------------- devices --

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    int max_pairs = 0;  // co-resident CTA pairs for the 2-CTA kernel
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

// ---------------------------------------------------------------- plans --

struct Plan {
    int variant = 0;
    int cta_group = 1;
    int arows = 128;       // A rows loaded per CTA (64: M <= 64, narrow kernel)
    int swap = 0;          // 1: the launch computes C^T = B^T A^T (M and N, A and B exchanged)
    int grid_m = 0, grid_n = 0;
    int bm = 128, bn = 256;
    int tiles_m = 0, tiles_n = 0, num_kb = 0;
    int grid = 0;
    int group_m = 1;
    int tiles_dp = 0, sk_tiles = 0;
    int64_t sk_iters = 0;
    uint32_t smem = 0;
    uint64_t slot_bytes = 0;  // workspace bytes per stream-K partial piece
    uint64_t ws_bytes = 0;    // workspace this plan needs (0 without stream-K)
    int ks = 1;               // CTAs of a cluster that split each tile's k-blocks (2: variant 7)
    int hilbert = 0;          // visiting order: 0 grouped bands, k > 0 the Hilbert curve of a 2^k square
    int ns = 1;               // MMAs per K step sharing the A operand (2: two half-width MMAs)
    void* ws_ptr = nullptr;   // the workspace of this launch
};


// Pipeline depths: what fits in 227 KB of shared memory next to the 32 KB of
// epilogue staging.
constexpr int kStages1 = 4;     // 1-CTA: 4 x (16 KB A + 32 KB B) per CTA
constexpr int kStages2 = 6;     // 2-CTA: 6 x (16 KB A + 16 KB B) per CTA
constexpr int kStages2n = 6;    // 2-CTA, 224 wide: 6 x (16 KB A + 14 KB B) per CTA
constexpr int kStagesN64 = 8;   // 1-CTA narrow: 8 x (16 KB A + 8 KB B)
constexpr int kStagesN64h = 12; // 1-CTA narrow, M <= 64: 12 x (8 KB A + 8 KB B)
using Cfg1 = tcg::GemmCfg<1, 256, kStages1>;
using Cfg2 = tcg::GemmCfg<2, 256, kStages2>;
using Cfg2n = tcg::GemmCfg<2, 224, kStages2n>;
using CfgN64 = tcg::GemmCfg<1, 64, kStagesN64>;
using CfgN64h = tcg::GemmCfg<1, 64, kStagesN64h, 64>;
// The transposed product with 128-row x 128-column tiles and the K split over
// a 2-CTA cluster (64 < M <= 128): 6 x (16 KB + 16 KB) per CTA, next to the
// 32 KB that stages half of the fp32 tile for the peer.
constexpr int kStagesS128 = 6;
using CfgS128 = tcg::GemmCfg<1, 128, kStagesS128, 128, 0, 2>;
static_assert(CfgS128::kSmemBytes <= 227 * 1024, "shared memory");
// The transposed product on CTA pairs: 64-row A stages (8 KB) and half of the
// B tile per CTA: 16 x (8 + 4) KB for up to 64 rows of C, 12 x (8 + 8) KB up
// to 128.
constexpr int kStagesSP = 16;
constexpr int kStagesSP128 = 12;
using CfgSP = tcg::GemmCfg<2, 64, kStagesSP, 64>;
using CfgSP128 = tcg::GemmCfg<2, 128, kStagesSP128, 64>;
static_assert(CfgSP::kSmemBytes <= 227 * 1024 && CfgSP128::kSmemBytes <= 227 * 1024, "shared memory");

// Variant numbers that name a kernel (3 is unused).
bool variant_known(int v) { return v >= TCGEMM_VARIANT_AUTO && v <= TCGEMM_VARIANT_SWAP_PAIR && v != 3; }

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Visiting order of the tiles: TCGEMM_ORDER=grouped or =hilbert in the
// environment chooses one for every launch (for A/B measurements); unset,
// the default order below is used.
int order_override() {
    static const int v = [] {
        const char* s = std::getenv("TCGEMM_ORDER");
        if (s && std::strcmp(s, "hilbert") == 0) return 1;
        if (s && std::strcmp(s, "grouped") == 0) return 0;
        return -1;
    }();
    return v;
}
constexpr bool kHilbertDefault = false;

// MMAs per K step for the CTA-pair tiles: TCGEMM_NSPLIT=1 or =2 in the
// environment chooses for every launch (A/B measurements); unset, 1.
int nsplit_choice() {
    static const int v = [] {
        const char* s = std::getenv("TCGEMM_NSPLIT");
        return (s && s[0] == '2') ? 2 : 1;
    }();
    return v;
}

// TCGEMM_SPLIT=0 in the environment turns the tail split off (for A/B timing).
bool split_enabled() {
    static const bool on = [] {
        const char* s = std::getenv("TCGEMM_SPLIT");
        return !(s && s[0] == '0');
    }();
    return on;
}

bool use_stream_k(int64_t tiles, int64_t clusters, int64_t num_kb);

// Estimated microseconds of a persistent launch (the variable part): rounds
// of tiles (or a stream-K share) times k-blocks times the time per k-block,
// which is the larger of the MMA's and the time to bring the k-block's
// operand bytes into the SM.  Measured on GB300: an SM receives operands at
// about 100 GB/s from L2 when every SM streams at once, the SM clock runs
// near 1.9 GHz, and a launch costs about 12 us (CTA pairs) or 10 us (single
// CTAs) on top (pipeline fill, last epilogue, launch).
double est_launch_us(int64_t tiles, int64_t units, int64_t num_kb, double mma_cycles_per_kb, double bytes_per_kb) {
    constexpr double kClockGHz = 1.9, kBytesPerUs = 100e3;
    const bool sk = use_stream_k(tiles, units, num_kb);
    const double kbs = sk ? static_cast<double>(tiles * num_kb) / static_cast<double>(units)
                          : static_cast<double>((tiles + units - 1) / units * num_kb);
    const double per_kb = std::max(mma_cycles_per_kb / (kClockGHz * 1e3), bytes_per_kb / kBytesPerUs);
    return kbs * per_kb + (sk ? 3.0 : 0.0);
}

// Automatic variant.  Up to 64 rows the product is computed transposed
// (C^T = B^T A^T), so that B's columns fill all 128 MMA rows and A's rows
// become the MMA's N; up to 128 rows the narrow 128 x 64 tiles give every SM
// its own columns of B.  Above that, CTA pairs (256-row tiles, M = 256 MMAs)
// unless the narrow tiles spread a small problem over many more SMs by
// enough to win: for 1024^3 they take 13.6 us against 17.1 us, for 2048^3
// 47.5 us against 24.2 us (GB300).  in_kind 1: 8-bit operands (a k-block of
// 128 values, the MMA twice as fast).
int pick_variant(int64_t M, int64_t N, int64_t K, int sms, int in_kind = 0) {
    if (M <= 128 && N >= 256) {
        // The transposed product (B's columns fill the 128 MMA rows).  When
        // its 128-row tiles fill between three quarters of a round and a
        // whole round of 2-CTA clusters, each tile's k-blocks are split over
        // the two CTAs of a cluster (no reduction pass); otherwise, up to 64
        // rows, stream-K shares them out when it pays.
        const int64_t tiles = (N + 127) / 128;
        const int64_t num_kb = (K + (in_kind == 1 ? 127 : 63)) / (in_kind == 1 ? 128 : 64);
        if (num_kb >= 8 && 2 * tiles <= sms && 8 * tiles >= 3 * static_cast<int64_t>(sms))
            return TCGEMM_VARIANT_SWAP_N64_KS2;
        if (M <= 64) return TCGEMM_VARIANT_SWAP_N64;
    }
    if (M <= 128) return TCGEMM_VARIANT_1CTA_N64;
    const int64_t num_kb = (K + (in_kind == 1 ? 127 : 63)) / (in_kind == 1 ? 128 : 64);
    const double mma_scale = in_kind == 1 ? 0.5 : 1.0;
    const int64_t pairs = std::max(1, sms / 2);
    double pair_us = 1e300;
    for (int64_t bn : {224, 256}) {
        const int64_t tiles = (M + 255) / 256 * ((N + bn - 1) / bn);
        pair_us = std::min(pair_us, est_launch_us(tiles, pairs, num_kb, 2.0 * bn * mma_scale, (128 + bn / 2) * 128.0));
    }
    const int64_t n64_tiles = (M + 127) / 128 * ((N + 63) / 64);
    const double n64_us = est_launch_us(n64_tiles, std::max(1, sms), num_kb, 128.0 * mma_scale, 192 * 128.0);
    return n64_us + 10.0 < pair_us + 12.0 ? TCGEMM_VARIANT_1CTA_N64 : TCGEMM_VARIANT_2CTA;
}

// Stream-K sharing: a piece pays the same fixed costs as a whole tile
// (pipeline fill, epilogue) and needs a reduction pass, so it only pays off
// when whole tiles would leave most clusters idle for a long mainloop: all
// tiles fit in half a round, K is at least 4096 (64 k-blocks), and every
// cluster still gets at least 4 k-blocks.  (Measured on GB300: 512x512x16384
// 80 -> 35 us, 256x2048x8192 46 -> 31 us; 1024x1280x2048 is faster without.)
bool use_stream_k(int64_t tiles, int64_t clusters, int64_t num_kb) {
    return 2 * tiles <= clusters && num_kb >= 64 && tiles * num_kb >= 4 * clusters;
}

// in_kind 0: bf16 operands (64 per k-block); 1: 8-bit operands (128 per k-block).
bool make_plan(int64_t M, int64_t N, int64_t K, int variant, int sms, int max_pairs, Plan& pl,
               bool allow_split = true, int in_kind = 0, bool a_col = false, bool b_row = false) {
    if (sms <= 0) return false;
    if (variant == TCGEMM_VARIANT_AUTO) variant = pick_variant(M, N, K, sms, in_kind);
    pl.variant = variant;
    allow_split = allow_split && split_enabled();
    if (variant == TCGEMM_VARIANT_SWAP_N64 || variant == TCGEMM_VARIANT_SWAP_N64_KS2 ||
        variant == TCGEMM_VARIANT_SWAP_PAIR) {
        // The transposed product: its M is N, its N is M.
        pl.swap = 1;
        std::swap(M, N);
    }
    const int64_t bk = in_kind == 1 ? 128 : 64;
    const int64_t num_kb = (K + bk - 1) / bk;
    if (variant == TCGEMM_VARIANT_1CTA) {
        pl.cta_group = 1;
        pl.bm = Cfg1::kBM;
        pl.bn = 256;
        pl.smem = Cfg1::kSmemBytes;
    } else if (variant == TCGEMM_VARIANT_2CTA || variant == TCGEMM_VARIANT_2CTA_W256) {
        pl.cta_group = 2;
        pl.bm = Cfg2::kBM;
        // Tile width 256 or 224, whichever is estimated to finish sooner.
        // Time per k-block ~ width + 32 (the shared-memory bytes a unit moves:
        // its A tile whatever the width, plus the B tile); k-blocks per cluster
        // = a balanced share with stream-K, else whole rounds of tiles.
        const int64_t pairs = std::max(1, max_pairs > 0 ? max_pairs : sms / 2);
        const int64_t tm = (M + 255) / 256;
        auto cost = [&](int64_t bn) {
            const int64_t t = tm * ((N + bn - 1) / bn);
            const double kbs = (allow_split && use_stream_k(t, pairs, num_kb))
                                   ? static_cast<double>(t * num_kb) / static_cast<double>(pairs)
                                   : static_cast<double>((t + pairs - 1) / pairs * num_kb);
            return kbs * static_cast<double>(bn + 32);
        };
        // An MN-major B tile is loaded in 64-value boxes: 112 per CTA does
        // not fit, so it takes the 256 width.
        pl.bn = (variant == TCGEMM_VARIANT_2CTA && !b_row && cost(224) < cost(256) * 0.97) ? 224 : 256;
        pl.smem = pl.bn == 224 ? Cfg2n::kSmemBytes : Cfg2::kSmemBytes;
    } else if (variant == TCGEMM_VARIANT_1CTA_N64 || variant == TCGEMM_VARIANT_SWAP_N64 ||
               variant == TCGEMM_VARIANT_SWAP_N64_KS2) {
        pl.cta_group = 1;
        pl.bm = CfgN64::kBM;
        pl.bn = 64;
        // Each CTA of the cluster needs at least one k-block.
        if (variant == TCGEMM_VARIANT_SWAP_N64_KS2 && num_kb >= 2) pl.ks = 2;
        pl.arows = (!pl.swap && M <= 64) ? 64 : 128;
        pl.smem = pl.arows == 64 ? CfgN64h::kSmemBytes : CfgN64::kSmemBytes;
        if (pl.ks == 2 && N > 64) {
            // More than 64 rows of C (the transposed product's N): 128-wide tiles.
            pl.bn = 128;
            pl.smem = CfgS128::kSmemBytes;
        }
    } else if (variant == TCGEMM_VARIANT_SWAP_PAIR) {
        // Here M is C's N and N is C's M (at most 128 rows of C).
        if (N > 128 || a_col || b_row || in_kind != 0) return false;
        pl.cta_group = 2;
        pl.bn = N <= 64 ? 64 : 128;
        // r rows per CTA: the smallest multiple of 8 that covers M with one
        // tile of 2r rows per resident pair, at most the 64-row stage.
        const int64_t pairs = std::max(1, max_pairs > 0 ? max_pairs : sms / 2);
        const int64_t r = std::min<int64_t>(64, std::max<int64_t>(8, (ceil_div(M, 2 * pairs) + 7) / 8 * 8));
        pl.arows = static_cast<int>(r);
        pl.bm = static_cast<int>(2 * r);
        pl.smem = pl.bn == 64 ? CfgSP::kSmemBytes : CfgSP128::kSmemBytes;
        allow_split = false;
    } else {
        return false;
    }
    pl.tiles_m = ceil_div(M, pl.bm);
    pl.tiles_n = ceil_div(N, pl.bn);
    pl.num_kb = static_cast<int>(num_kb);
    pl.slot_bytes = static_cast<uint64_t>(pl.cta_group) * 128 * pl.bn * 4;
    pl.grid_m = pl.tiles_m;
    pl.grid_n = pl.tiles_n;
    const int64_t tiles = static_cast<int64_t>(pl.grid_m) * pl.grid_n;  // units of the order
    if (tiles > (int64_t{1} << 30)) return false;
    int64_t clusters = sms;
    if (pl.cta_group == 2 || pl.ks == 2) clusters = std::max(1, max_pairs > 0 ? max_pairs : sms / 2);
    if (pl.ks == 2) allow_split = false;  // the split is the cluster's
    const int csize = pl.cta_group * pl.ks;
    pl.tiles_dp = static_cast<int>(tiles);
    pl.sk_tiles = 0;
    pl.sk_iters = 0;
    if (allow_split && use_stream_k(tiles, clusters, num_kb)) {
        const int64_t rem = tiles % clusters;
        pl.sk_tiles = static_cast<int>(rem);
        pl.sk_iters = rem * num_kb;
        pl.tiles_dp = static_cast<int>(tiles - rem);
        pl.grid = static_cast<int>(clusters) * csize;
        // Two partial slots per cluster (the first and last segment of its range).
        pl.ws_bytes = 2 * static_cast<uint64_t>(clusters) * pl.slot_bytes;
    } else {
        pl.grid = static_cast<int>(std::min<int64_t>(tiles, clusters)) * csize;
        pl.ws_bytes = 0;
    }
    // Band height so that the tiles in flight at once cover a roughly square
    // patch of C: group_m^2 ~ concurrent tiles * (tile width / tile height).
    // Pair tiles take a band twice that tall (measured on GB300: 16 instead
    // of 8 rows of tiles, 4000x4100x4104 110.5 -> 108.3 us, 16384x8192x4096
    // 594 -> 584 us, the square shapes unchanged): B is fetched from memory
    // once per band, so fewer bands re-read it less often.
    const double ideal = std::sqrt(static_cast<double>(pl.grid / csize) * pl.bn / pl.bm) *
                         (pl.cta_group == 2 ? 2.0 : 1.0);
    int g = 1;
    while (g * 2 <= ideal) g *= 2;
    pl.group_m = std::max(1, std::min(g, pl.grid_m));
    if (in_kind == 0 && ((pl.cta_group == 2 && !pl.swap) || (pl.swap && pl.ks == 2 && pl.bn == 64)))
        pl.ns = nsplit_choice();
    const int ov = order_override();
    if (ov == 1 || (ov < 0 && kHilbertDefault)) {
        int k = 0;
        while ((1 << k) < std::max(pl.grid_m, pl.grid_n)) ++k;
        pl.hilbert = k;  // 0 for a single tile: the two orders agree
    }
    return true;
}

// --------------------------------------------------------- tensor maps --

// C (column-major M x N, fp32, bf16 or int8) in boxes of box_rows rows x 32
// columns: 32-row boxes for the epilogue warps' TMA loads, stores and L2
// prefetches of C; 128-row boxes for the stream-K workspace (fp32, 128 rows,
// ldc = 128).
bool encode_c(CUtensorMap* m, void* ptr, int64_t M, int64_t N, int64_t ldc, int out_dtype, uint32_t box_rows) {
    if (!encode_fn()) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    const uint64_t esz = out_dtype == TCGEMM_OUT_F32 ? 4 : out_dtype == TCGEMM_OUT_BF16 ? 2 : 1;
    const CUtensorMapDataType dt = out_dtype == TCGEMM_OUT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : out_dtype == TCGEMM_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                  : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const MapKey k{dt, ptr, {static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(N)},
                   static_cast<cuuint64_t>(ldc) * esz, {box_rows, 32u}, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE};
    const CUresult r = encode_2d(m, k);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d) for C %lld x %lld, ldc %lld", static_cast<int>(r),
                  static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(ldc));
        return false;
    }
    return true;
}

bool encode_kmajor(CUtensorMap* m, const void* ptr, int64_t k_extent, int64_t rows, int64_t ld,
                   uint32_t box_rows, int elem_bytes = 2) {
    if (!encode_fn()) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    // One 128-byte row per box row: 64 bf16 or 128 8-bit values.  No L2
    // promotion: where rows are not 128-byte aligned a box row touches two
    // lines, and promoting each miss to 256 bytes fetches bytes no box uses
    // (4000x4100x4104: 115 -> 106 us; aligned shapes unchanged).
    const MapKey k{elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr,
                   {static_cast<cuuint64_t>(k_extent), static_cast<cuuint64_t>(rows)},
                   static_cast<cuuint64_t>(ld) * static_cast<cuuint64_t>(elem_bytes),
                   {128u / static_cast<cuuint32_t>(elem_bytes), box_rows}, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE};
    const CUresult r = encode_2d(m, k);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d) for extent %lld x %lld, ld %lld", static_cast<int>(r),
                  static_cast<long long>(k_extent), static_cast<long long>(rows), static_cast<long long>(ld));
        return false;
    }
    return true;
}

// An MN-major operand (M or N contiguous; bf16): dims {MN, K}, boxes of 64
// MN values (one 128-byte swizzled row) by 64 K rows.
bool encode_mnmajor(CUtensorMap* m, const void* ptr, int64_t mn_extent, int64_t k_extent, int64_t ld) {
    if (!encode_fn()) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    const MapKey k{CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr,
                   {static_cast<cuuint64_t>(mn_extent), static_cast<cuuint64_t>(k_extent)},
                   static_cast<cuuint64_t>(ld) * 2u, {64u, 64u}, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B};
    const CUresult r = encode_2d(m, k);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d) for an MN-major operand %lld x %lld, ld %lld",
                  static_cast<int>(r), static_cast<long long>(mn_extent), static_cast<long long>(k_extent),
                  static_cast<long long>(ld));
        return false;
    }
    return true;
}

// -------------------------------------------------------------- launch --

// The dynamic shared-memory opt-in is a per-kernel attribute; it is set once
// per device for each kernel instantiation.
template <int CG, int BN, int ST, int AR, bool SW, typename OutT, int IN = 0, int KS = 1, int NS = 1>
bool ensure_smem_attr(int dev) {
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    std::lock_guard<std::mutex> lk(mu);
    if (done[dev]) return true;
    auto kern = tcg::gemm_bf16_tn_kernel<CG, BN, ST, AR, SW, OutT, IN, KS, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(tcg::GemmCfg<CG, BN, ST, AR, IN, KS>::kSmemBytes));
    if (e != cudaSuccess) {
        set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return false;
    }
    done[dev] = true;
    return true;
}

template <int CG, int BN, int ST, int AR, bool SW, typename OutT, int IN = 0, int KS = 1, int NS = 1>
int launch_gemm(const Plan& pl, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tcm,
                const CUtensorMap& twm, const tcg::GemmParams& gp, cudaStream_t stream, int dev) {
    auto kern = tcg::gemm_bf16_tn_kernel<CG, BN, ST, AR, SW, OutT, IN, KS, NS>;
    if (!ensure_smem_attr<CG, BN, ST, AR, SW, OutT, IN, KS, NS>(dev)) return TCGEMM_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.grid), 1, 1);
    cfg.blockDim = dim3(tcg::GemmCfg<CG, BN, ST, AR>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    // A programmatic dependent of the previous kernel on the stream: the
    // launch and the set-up (barriers, TMEM, the first unit) overlap that
    // kernel's tail; the kernel reads no global memory before it completes.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (CG * KS > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = CG * KS;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tcm, twm, gp);
    if (e != cudaSuccess) {
        set_error("kernel launch: %s", cudaGetErrorString(e));
        return TCGEMM_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (pl.sk_tiles > 0) {
        // Add up the shared tiles' partials (same stream, so after the GEMM).
        const unsigned blocks = static_cast<unsigned>(pl.sk_tiles * tcg::sk_reduce_blocks_per_tile<CG, BN>());
        cudaLaunchConfig_t rcfg = {};
        rcfg.gridDim = dim3(blocks, 1, 1);
        rcfg.blockDim = dim3(128, 1, 1);
        rcfg.stream = stream;
        cudaLaunchAttribute rattr[1];
        rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        rattr[0].val.programmaticStreamSerializationAllowed = 1;
        rcfg.attrs = rattr;
        rcfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&rcfg, tcg::sk_reduce_kernel<CG, BN, SW, OutT>, static_cast<const float*>(pl.ws_ptr),
                               gp, pl.grid / CG);
        if (e != cudaSuccess) {
            set_error("reduction kernel launch: %s", cudaGetErrorString(e));
            return TCGEMM_ERR_CUDA;
        }
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    return TCGEMM_OK;
}

template <typename Kern>
int max_active_clusters(Kern kern, int cluster, uint32_t smem, int sms) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms / cluster * cluster), 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    (void)cudaGetLastError();
    return n;
}

int probe_device(int& dev_out, DeviceInfo& info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("cudaGetDevice: %s", cudaGetErrorString(e));
        return TCGEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("device ordinal %d out of range", dev);
        return TCGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    dev_out = dev;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        d.supported = (major == 10 && minor == 3);
        d.sms = sms;
        d.max_pairs = sms / 2;
        if (d.supported) {
            // How many clusters of each kind can be resident at once (cluster
            // placement may leave some SMs of a GPC unused).
            if (ensure_smem_attr<2, 256, kStages2, 128, false, __nv_bfloat16>(dev)) {
                const int n = max_active_clusters(tcg::gemm_bf16_tn_kernel<2, 256, kStages2, 128, false, __nv_bfloat16>,
                                                  2, Cfg2::kSmemBytes, sms);
                if (n > 0) d.max_pairs = n;
            }
        }
        d.probed = true;
    }
    info = d;
    if (!d.supported) {
        set_error("device %d is not compute capability 10.3 (sm_103a)", dev);
        return TCGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    return TCGEMM_OK;
}

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    const uintptr_t a1 = a0 + static_cast<uintptr_t>(abytes), b1 = b0 + static_cast<uintptr_t>(bbytes);
    return a0 < b1 && b0 < a1;
}

int validate(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
             const void* C, int64_t ldc, int out_dtype, int64_t in_bytes = 2, bool a_col = false,
             bool b_row = false) {
    const int64_t lim = (int64_t{1} << 31) - 1;
    if (M < 0 || N < 0 || K < 0 || M > lim || N > lim || K > lim) {
        set_error("sizes must satisfy 0 <= M, N, K < 2^31 (got %lld, %lld, %lld)", static_cast<long long>(M),
                  static_cast<long long>(N), static_cast<long long>(K));
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (out_dtype != TCGEMM_OUT_F32 && out_dtype != TCGEMM_OUT_BF16 && out_dtype != TCGEMM_OUT_I8) {
        set_error("out_dtype must be TCGEMM_OUT_F32 (0), TCGEMM_OUT_BF16 (1) or TCGEMM_OUT_I8 (2), got %d",
                  out_dtype);
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (lda < std::max<int64_t>(a_col ? M : K, 1) || ldb < std::max<int64_t>(b_row ? N : K, 1) ||
        ldc < std::max<int64_t>(M, 1)) {
        set_error("leading dimensions too small: need lda >= %s, ldb >= %s, ldc >= M (at least 1)",
                  a_col ? "M" : "K", b_row ? "N" : "K");
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (M == 0 || N == 0) return TCGEMM_OK;
    const int64_t esz = out_dtype == TCGEMM_OUT_F32 ? 4 : out_dtype == TCGEMM_OUT_BF16 ? 2 : 1;
    if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))) {
        set_error("null matrix pointer");
        return TCGEMM_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 || ((ldc * esz) & 15) != 0) {
        set_error("C must be 16-byte aligned with ldc*%lld a multiple of 16 bytes", static_cast<long long>(esz));
        return TCGEMM_ERR_ALIGNMENT;
    }
    if (K > 0) {
        if ((reinterpret_cast<uintptr_t>(A) & 15u) != 0 || (reinterpret_cast<uintptr_t>(B) & 15u) != 0 ||
            ((lda * in_bytes) & 15) != 0 || ((ldb * in_bytes) & 15) != 0) {
            set_error("A and B must be 16-byte aligned with lda and ldb multiples of 16 bytes (%lld-byte elements)",
                      static_cast<long long>(in_bytes));
            return TCGEMM_ERR_ALIGNMENT;
        }
        const int64_t cbytes = ((N - 1) * ldc + M) * esz;
        const int64_t a_elems = a_col ? (K - 1) * lda + M : (M - 1) * lda + K;
        const int64_t b_elems = b_row ? (K - 1) * ldb + N : (N - 1) * ldb + K;
        if (overlaps(C, cbytes, A, a_elems * in_bytes) || overlaps(C, cbytes, B, b_elems * in_bytes)) {
            set_error("C overlaps A or B");
            return TCGEMM_ERR_INVALID_ARG;
        }
    }
    return TCGEMM_OK;
}

// Largest workspace any plan on a device with `sms` SMs can need: two partial
// slots per cluster, 128 rows x 256 columns of fp32 per CTA.
uint64_t max_workspace_bytes(int sms) { return 2 * static_cast<uint64_t>(sms) * 128 * 256 * 4; }

// Library-owned split workspace, one per (device, stream) so that calls on
// different streams never share partials.  Allocated the first time a
// stream-K plan runs on that stream.
struct InternalWs {
    void* ptr = nullptr;
    uint64_t bytes = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, InternalWs> g_ws;

int internal_workspace(int dev, int sms, cudaStream_t stream, uint64_t need, void** out) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    InternalWs& w = g_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (w.bytes < need) {
        const uint64_t bytes = std::max(need, max_workspace_bytes(sms));
        void* p = nullptr;
        cudaError_t e = cudaMalloc(&p, bytes);
        if (e != cudaSuccess) {
            set_error("workspace cudaMalloc(%llu): %s", static_cast<unsigned long long>(bytes), cudaGetErrorString(e));
            return TCGEMM_ERR_CUDA;
        }
        if (w.ptr) cudaFree(w.ptr);  // never reached in practice: the first block is the maximum
        w.ptr = p;
        w.bytes = bytes;
    }
    *out = w.ptr;
    return TCGEMM_OK;
}

// ---------------------------------------------- fixed scratch, no allocation --
//
// Scratch for gemm_bf16_noalloc: a file-scope device array of fixed size, so
// that entry point never allocates.  Every GPU that loads this library holds
// these 40 MiB until the process exits.  In host code the array's name is only
// a stand-in: its device address comes from cudaGetSymbolAddress, taken once
// per device (with that device current) on the first call there.
constexpr uint64_t kNoAllocScratchBytes = uint64_t{40} << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The fixed array holds a plan's workspace.
bool noalloc_fits(uint64_t ws_bytes) { return ws_bytes <= kNoAllocScratchBytes; }

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            set_error("cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
            return TCGEMM_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return TCGEMM_OK;
}

void fill_plan_out(const Plan& pl, int64_t* out) {
    out[0] = pl.grid;
    out[1] = pl.cta_group * pl.ks;
    out[2] = pl.tiles_m;
    out[3] = pl.tiles_n;
    out[4] = pl.bm;
    out[5] = pl.bn;
    out[6] = pl.num_kb;
    out[7] = pl.smem;
    out[8] = pl.tiles_dp;
    out[9] = pl.sk_tiles;
    out[10] = pl.sk_iters;
    out[11] = static_cast<int64_t>(pl.ws_bytes);
    out[12] = pl.group_m;
    out[13] = pl.variant;
    out[14] = pl.cta_group;
    out[15] = pl.grid_m;
    out[16] = pl.grid_n;
    out[17] = pl.sk_tiles > 0 ? 1 : 0;
    out[18] = pl.arows;
    out[19] = pl.swap;
    out[20] = pl.ks;
    out[21] = pl.hilbert;
}

constexpr int kWsInternal = 0;
constexpr int kWsCaller = 1;
constexpr int kWsNone = 2;     // plan without any split
constexpr int kWsNoAlloc = 3;  // the fixed scratch array above

// The fused epilogue of one call: bias (one value per column of C) and
// activation; the default is none of either.
struct Epilogue {
    const void* bias = nullptr;
    int bias_kind = TCGEMM_BIAS_NONE;
    int act = TCGEMM_ACT_NONE;
    const float* qscale = nullptr;  // int8 output: one scale per row of C
    int qzero = 0;                  // int8 output: zero point
};

int validate_epilogue(const Epilogue& ep, int64_t M, int64_t N, const void* C, int64_t ldc, int out_dtype) {
    if (ep.act < TCGEMM_ACT_NONE || ep.act > TCGEMM_ACT_GELU_TANH) {
        set_error("unknown activation %d", ep.act);
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (ep.bias_kind < TCGEMM_BIAS_NONE || ep.bias_kind > TCGEMM_BIAS_BF16) {
        set_error("unknown bias dtype %d", ep.bias_kind);
        return TCGEMM_ERR_INVALID_ARG;
    }
    if ((ep.bias_kind == TCGEMM_BIAS_NONE) != (ep.bias == nullptr)) {
        set_error("bias must be NULL exactly when bias_dtype is TCGEMM_BIAS_NONE");
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (out_dtype == TCGEMM_OUT_I8) {
        if (ep.qscale == nullptr) {
            set_error("int8 output needs the per-row scales (gemm_quant_i8)");
            return TCGEMM_ERR_INVALID_ARG;
        }
        if ((reinterpret_cast<uintptr_t>(ep.qscale) & 15u) != 0) {
            set_error("row_scale must be 16-byte aligned");
            return TCGEMM_ERR_ALIGNMENT;
        }
        if (M > 0 && N > 0 &&
            overlaps(C, ((N - 1) * ldc + M), ep.qscale, M * static_cast<int64_t>(sizeof(float)))) {
            set_error("row_scale overlaps the output");
            return TCGEMM_ERR_INVALID_ARG;
        }
    }
    if (ep.bias_kind == TCGEMM_BIAS_NONE || M == 0 || N == 0) return TCGEMM_OK;
    const int64_t besz = ep.bias_kind == TCGEMM_BIAS_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(ep.bias) & static_cast<uintptr_t>(besz - 1)) != 0) {
        set_error("bias must be aligned to its element size (%lld bytes)", static_cast<long long>(besz));
        return TCGEMM_ERR_ALIGNMENT;
    }
    const int64_t esz = out_dtype == TCGEMM_OUT_F32 ? 4 : out_dtype == TCGEMM_OUT_BF16 ? 2 : 1;
    if (overlaps(C, ((N - 1) * ldc + M) * esz, ep.bias, N * besz)) {
        set_error("bias overlaps C");
        return TCGEMM_ERR_INVALID_ARG;
    }
    return TCGEMM_OK;
}

// ------------------------------------------------------------ autotuning --

// The variant measured fastest for a problem, per device: filled by
// tcgemm_autotune, consulted by every call that asks for the automatic
// choice.
struct TuneKey {
    int dev;
    int64_t M, N, K;
    int in_kind, in_fmt, out_dtype, a_col, b_row, has_beta;
    bool operator<(const TuneKey& o) const {
        return std::tie(dev, M, N, K, in_kind, in_fmt, out_dtype, a_col, b_row, has_beta) <
               std::tie(o.dev, o.M, o.N, o.K, o.in_kind, o.in_fmt, o.out_dtype, o.a_col, o.b_row, o.has_beta);
    }
};
std::mutex g_tune_mu;
std::map<TuneKey, int> g_tuned;

int tuned_variant(const TuneKey& k) {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    auto it = g_tuned.find(k);
    return it == g_tuned.end() ? TCGEMM_VARIANT_AUTO : it->second;
}

int run_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
             int64_t ldc, float alpha, float beta, int out_dtype, void* stream_v, int variant,
             int ws_mode = kWsInternal, void* ws = nullptr, int64_t ws_bytes = 0, const Epilogue& ep = Epilogue(),
             int in_kind = 0, int in_fmt = 0, bool a_col = false, bool b_row = false, int withhold_kb = -1,
             uint64_t timeout_override_ns = 0, int in_fmt_b = -1) {
    t_last_error[0] = '\0';
    if (!variant_known(variant)) {
        set_error("unknown variant %d", variant);
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (in_kind == 1) {
        if (in_fmt_b < 0) in_fmt_b = in_fmt;  // both operands in one format
        if ((in_fmt != TCGEMM_FP8_E4M3 && in_fmt != TCGEMM_FP8_E5M2) ||
            (in_fmt_b != TCGEMM_FP8_E4M3 && in_fmt_b != TCGEMM_FP8_E5M2)) {
            set_error("unknown FP8 format %d / %d", in_fmt, in_fmt_b);
            return TCGEMM_ERR_INVALID_ARG;
        }
        if (variant == TCGEMM_VARIANT_1CTA || variant == TCGEMM_VARIANT_SWAP_PAIR) {
            set_error("variant %d is not built for FP8 operands", variant);
            return TCGEMM_ERR_INVALID_ARG;
        }
    }
    if (out_dtype == TCGEMM_OUT_I8) {
        if (beta != 0.0f) {
            set_error("int8 output is written only: beta must be 0");
            return TCGEMM_ERR_INVALID_ARG;
        }
        if (variant == TCGEMM_VARIANT_1CTA || variant == TCGEMM_VARIANT_SWAP_PAIR) {
            set_error("variant %d is not built for int8 output", variant);
            return TCGEMM_ERR_INVALID_ARG;
        }
    }
    if ((a_col || b_row) && in_kind == 1) {
        set_error("column-major A / row-major B: bf16 operands only");
        return TCGEMM_ERR_INVALID_ARG;
    }
    int rc = validate(M, N, K, A, lda, B, ldb, C, ldc, out_dtype, in_kind == 1 ? 1 : 2, a_col, b_row);
    if (rc != TCGEMM_OK) return rc;
    rc = validate_epilogue(ep, M, N, C, ldc, out_dtype);
    if (rc != TCGEMM_OK) return rc;
    if (M == 0 || N == 0) return TCGEMM_OK;
    int dev = 0;
    DeviceInfo info;
    rc = probe_device(dev, info);
    if (rc != TCGEMM_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    // The tuned-choice table holds problems whose operands share one format.
    if (variant == TCGEMM_VARIANT_AUTO && (in_kind == 0 || in_fmt_b == in_fmt)) {
        const TuneKey key{dev, M, N, K, in_kind, in_kind == 1 ? in_fmt : 0, out_dtype, a_col ? 1 : 0, b_row ? 1 : 0,
                          beta != 0.0f ? 1 : 0};
        variant = tuned_variant(key);
    }

    if (K == 0) {
        const int64_t total = M * N;
        const int threads = 256;
        const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, int64_t{info.sms} * 8);
        tcg::GemmParams sp{};
        sp.M = static_cast<int>(M);
        sp.N = static_cast<int>(N);
        sp.ldc = ldc;
        sp.C = C;
        sp.alpha = alpha;
        sp.beta = beta;
        sp.bias = ep.bias;
        sp.bias_kind = ep.bias_kind;
        sp.act = ep.act;
        sp.qscale = ep.qscale;
        sp.qzero = static_cast<float>(ep.qzero);
        if (out_dtype == TCGEMM_OUT_F32) {
            tcg::scale_c_kernel<float><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(sp);
        } else if (out_dtype == TCGEMM_OUT_I8) {
            tcg::scale_c_kernel<int8_t><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(sp);
        } else {
            tcg::scale_c_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(sp);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error("kernel launch: %s", cudaGetErrorString(e));
            return TCGEMM_ERR_CUDA;
        }
        g_launches.fetch_add(1, std::memory_order_relaxed);
        return TCGEMM_OK;
    }

    Plan pl;
    if (!make_plan(M, N, K, variant, info.sms, info.max_pairs, pl, ws_mode != kWsNone, in_kind,
                   a_col, b_row)) {
        set_error("no launch plan for this shape and variant");
        return TCGEMM_ERR_INVALID_ARG;
    }
    void* wsp = nullptr;
    if (pl.ws_bytes > 0) {
        if (ws_mode == kWsCaller) {
            if (ws == nullptr || ws_bytes < 0 || static_cast<uint64_t>(ws_bytes) < pl.ws_bytes ||
                (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) {
                set_error("workspace must be 256-byte aligned and hold %llu bytes",
                          static_cast<unsigned long long>(pl.ws_bytes));
                return TCGEMM_ERR_INVALID_ARG;
            }
            wsp = ws;
        } else if (ws_mode == kWsNoAlloc) {
            if (!noalloc_fits(pl.ws_bytes)) {
                set_error("this shape needs %llu bytes of scratch, more than the fixed %llu of gemm_bf16_noalloc",
                          static_cast<unsigned long long>(pl.ws_bytes),
                          static_cast<unsigned long long>(kNoAllocScratchBytes));
                return TCGEMM_ERR_INVALID_ARG;
            }
            // The array keeps the last call's contents; every partial is
            // written before it is read, so nothing needs clearing.
            rc = noalloc_scratch(dev, &wsp);
            if (rc != TCGEMM_OK) return rc;
        } else {
            rc = internal_workspace(dev, info.sms, static_cast<cudaStream_t>(stream_v), pl.ws_bytes, &wsp);
            if (rc != TCGEMM_OK) return rc;
        }
    }
    // The split-MMA kernels are built for bf16 operands with fp32 or bf16
    // output; the others issue one MMA per K step.
    if (out_dtype == TCGEMM_OUT_I8) pl.ns = 1;
    // Box heights: a CTA pair loads half of the B tile per CTA (in pl.ns
    // boxes).
    const uint32_t a_box_rows = (pl.arows == 64 || (pl.swap && pl.cta_group == 2)) ? static_cast<uint32_t>(pl.arows)
                                                                                    : 128u;
    const uint32_t b_box_rows = static_cast<uint32_t>(pl.cta_group == 2 ? pl.bn / 2 / pl.ns : pl.bn);
    // The transposed product multiplies B^T (N x K, rows of B contiguous in
    // k) by A^T: the operands trade places.
    const void* opA = pl.swap ? B : A;
    const void* opB = pl.swap ? A : B;
    const int64_t rowsA = pl.swap ? N : M, rowsB = pl.swap ? M : N;
    const int64_t ldA = pl.swap ? ldb : lda, ldB = pl.swap ? lda : ldb;
    // The MMA's A operand is A (B in the transposed product); MN-major when
    // that matrix is stored with its M (N) index contiguous.
    const bool mma_a_mn = pl.swap ? b_row : a_col, mma_b_mn = pl.swap ? a_col : b_row;
    CUtensorMap ta, tb;
    const int in_bytes = in_kind == 1 ? 1 : 2;
    const bool ok_a = mma_a_mn ? encode_mnmajor(&ta, opA, rowsA, K, ldA)
                               : encode_kmajor(&ta, opA, K, rowsA, ldA, a_box_rows, in_bytes);
    const bool ok_b = mma_b_mn ? encode_mnmajor(&tb, opB, rowsB, K, ldB)
                               : encode_kmajor(&tb, opB, K, rowsB, ldB, b_box_rows, in_bytes);
    if (!ok_a || !ok_b) {
        return TCGEMM_ERR_INVALID_ARG;
    }
    pl.ws_ptr = wsp;
    CUtensorMap tcm, twm;
    if (!encode_c(&tcm, C, M, N, ldc, out_dtype, 32u)) return TCGEMM_ERR_INVALID_ARG;
    if (pl.sk_tiles > 0) {
        const int64_t wcols = 2 * static_cast<int64_t>(pl.grid / pl.cta_group) * pl.cta_group * pl.bn;
        if (!encode_c(&twm, wsp, 128, wcols, 128, TCGEMM_OUT_F32, 128u))
            return TCGEMM_ERR_INVALID_ARG;
    } else {
        twm = tcm;
    }
    tcg::GemmParams gp{};
    gp.M = static_cast<int>(pl.swap ? N : M);
    gp.N = static_cast<int>(pl.swap ? M : N);
    gp.K = static_cast<int>(K);
    gp.tiles_m = pl.tiles_m;
    gp.tiles_n = pl.tiles_n;
    gp.num_kb = pl.num_kb;
    gp.group_m = pl.group_m;
    gp.hilbert = pl.hilbert;
    gp.grid_m = pl.grid_m;
    gp.grid_n = pl.grid_n;
    gp.ldc = ldc;
    gp.C = C;
    gp.alpha = alpha;
    gp.beta = beta;
    gp.bias = ep.bias;
    gp.bias_kind = ep.bias_kind;
    gp.act = ep.act;
    // The MMA's operand formats: A's and B's, exchanged in the transposed product.
    if (in_kind == 1) {
        const int fa = pl.swap ? in_fmt_b : in_fmt, fb = pl.swap ? in_fmt : in_fmt_b;
        gp.in_fmt = (fa & 1) | ((fb & 1) << 1);
    }
    gp.qscale = ep.qscale;
    gp.qzero = static_cast<float>(ep.qzero);
    gp.a_mn = mma_a_mn ? 1 : 0;
    gp.b_mn = mma_b_mn ? 1 : 0;
    gp.tiles_dp = pl.tiles_dp;
    gp.sk_tiles = pl.sk_tiles;
    gp.sk_iters = pl.sk_iters;
    gp.rows_a = pl.arows;
    gp.timeout_ns = timeout_override_ns > 0 ? timeout_override_ns : timeout_ns();
    gp.withhold_kb = withhold_kb;

    const bool bf16 = out_dtype == TCGEMM_OUT_BF16;
    if (out_dtype == TCGEMM_OUT_I8) {
        // The quantising epilogue: CTA-pair tiles, narrow tiles, the
        // transposed product; bf16 or 8-bit operands.
#define TCGEMM_LAUNCH_I8(CG, BN, ST, AR, SW)                                                             \
    return in_kind == 1 ? launch_gemm<CG, BN, ST, AR, SW, int8_t, 1>(pl, ta, tb, tcm, twm, gp, stream, dev) \
                        : launch_gemm<CG, BN, ST, AR, SW, int8_t, 0>(pl, ta, tb, tcm, twm, gp, stream, dev)
        if (pl.swap && pl.ks == 2 && pl.bn == 128)
            return in_kind == 1 ? launch_gemm<1, 128, kStagesS128, 128, true, int8_t, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                                : launch_gemm<1, 128, kStagesS128, 128, true, int8_t, 0, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
        if (pl.swap && pl.ks == 2)
            return in_kind == 1 ? launch_gemm<1, 64, kStagesN64, 128, true, int8_t, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                                : launch_gemm<1, 64, kStagesN64, 128, true, int8_t, 0, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
        if (pl.swap) TCGEMM_LAUNCH_I8(1, 64, kStagesN64, 128, true);
        if (pl.bn == 64 && pl.arows == 64) TCGEMM_LAUNCH_I8(1, 64, kStagesN64h, 64, false);
        if (pl.bn == 64) TCGEMM_LAUNCH_I8(1, 64, kStagesN64, 128, false);
        if (pl.cta_group == 2 && pl.bn == 224) TCGEMM_LAUNCH_I8(2, 224, kStages2n, 128, false);
        if (pl.cta_group == 2) TCGEMM_LAUNCH_I8(2, 256, kStages2, 128, false);
#undef TCGEMM_LAUNCH_I8
        set_error("no int8-output kernel for this plan");
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (in_kind == 1) {
        // 8-bit operands: the CTA-pair tiles, the narrow tiles and the
        // transposed product.
#define TCGEMM_LAUNCH8(CG, BN, ST, AR, SW)                                                                  \
    return bf16 ? launch_gemm<CG, BN, ST, AR, SW, __nv_bfloat16, 1>(pl, ta, tb, tcm, twm, gp, stream, dev) \
                : launch_gemm<CG, BN, ST, AR, SW, float, 1>(pl, ta, tb, tcm, twm, gp, stream, dev)
        if (pl.swap && pl.ks == 2 && pl.bn == 128)
            return bf16 ? launch_gemm<1, 128, kStagesS128, 128, true, __nv_bfloat16, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                        : launch_gemm<1, 128, kStagesS128, 128, true, float, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
        if (pl.swap && pl.ks == 2)
            return bf16 ? launch_gemm<1, 64, kStagesN64, 128, true, __nv_bfloat16, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                        : launch_gemm<1, 64, kStagesN64, 128, true, float, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
        if (pl.swap) TCGEMM_LAUNCH8(1, 64, kStagesN64, 128, true);
        if (pl.bn == 64 && pl.arows == 64) TCGEMM_LAUNCH8(1, 64, kStagesN64h, 64, false);
        if (pl.bn == 64) TCGEMM_LAUNCH8(1, 64, kStagesN64, 128, false);
        if (pl.cta_group == 2 && pl.bn == 224) TCGEMM_LAUNCH8(2, 224, kStages2n, 128, false);
        if (pl.cta_group == 2) TCGEMM_LAUNCH8(2, 256, kStages2, 128, false);
#undef TCGEMM_LAUNCH8
        set_error("no FP8 kernel for this plan");
        return TCGEMM_ERR_INVALID_ARG;
    }
#define TCGEMM_LAUNCH(CG, BN, ST, AR, SW)                                                               \
    return bf16 ? launch_gemm<CG, BN, ST, AR, SW, __nv_bfloat16>(pl, ta, tb, tcm, twm, gp, stream, dev) \
                : launch_gemm<CG, BN, ST, AR, SW, float>(pl, ta, tb, tcm, twm, gp, stream, dev)
    if (pl.swap && pl.cta_group == 2 && pl.bn == 128) TCGEMM_LAUNCH(2, 128, kStagesSP128, 64, true);
    if (pl.swap && pl.cta_group == 2) TCGEMM_LAUNCH(2, 64, kStagesSP, 64, true);
    if (pl.swap && pl.ks == 2 && pl.bn == 128)
        return bf16 ? launch_gemm<1, 128, kStagesS128, 128, true, __nv_bfloat16, 0, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                    : launch_gemm<1, 128, kStagesS128, 128, true, float, 0, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
    if (pl.swap && pl.ks == 2 && pl.ns == 2)
        return bf16 ? launch_gemm<1, 64, kStagesN64, 128, true, __nv_bfloat16, 0, 2, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                    : launch_gemm<1, 64, kStagesN64, 128, true, float, 0, 2, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
    if (pl.swap && pl.ks == 2)
        return bf16 ? launch_gemm<1, 64, kStagesN64, 128, true, __nv_bfloat16, 0, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                    : launch_gemm<1, 64, kStagesN64, 128, true, float, 0, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
    if (pl.swap) TCGEMM_LAUNCH(1, 64, kStagesN64, 128, true);
    if (pl.bn == 64 && pl.arows == 64) TCGEMM_LAUNCH(1, 64, kStagesN64h, 64, false);
    if (pl.bn == 64) TCGEMM_LAUNCH(1, 64, kStagesN64, 128, false);
    if (pl.cta_group == 1) TCGEMM_LAUNCH(1, 256, kStages1, 128, false);
    if (pl.bn == 224 && pl.ns == 2)
        return bf16 ? launch_gemm<2, 224, kStages2n, 128, false, __nv_bfloat16, 0, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                    : launch_gemm<2, 224, kStages2n, 128, false, float, 0, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
    if (pl.bn == 224) TCGEMM_LAUNCH(2, 224, kStages2n, 128, false);
    if (pl.ns == 2)
        return bf16 ? launch_gemm<2, 256, kStages2, 128, false, __nv_bfloat16, 0, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev)
                    : launch_gemm<2, 256, kStages2, 128, false, float, 0, 1, 2>(pl, ta, tb, tcm, twm, gp, stream, dev);
    TCGEMM_LAUNCH(2, 256, kStages2, 128, false);
#undef TCGEMM_LAUNCH
}

}  // namespace

extern "C" {

int gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
              int64_t ldc, float alpha, float beta, int out_dtype, void* stream) {
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, TCGEMM_VARIANT_AUTO);
}

int gemm_bf16_variant(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                      void* C, int64_t ldc, float alpha, float beta, int out_dtype, void* stream, int variant) {
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant);
}

int gemm_bf16_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                 int64_t ldc, float alpha, float beta, int out_dtype, void* stream, int variant, void* workspace,
                 int64_t workspace_bytes) {
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant, kWsCaller, workspace,
                    workspace_bytes);
}

int gemm_bf16_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                      void* C, int64_t ldc, float alpha, float beta, int out_dtype, void* stream, int variant) {
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant, kWsNoAlloc);
}

int gemm_bf16_bias_act(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                       void* C, int64_t ldc, float alpha, float beta, int out_dtype, const void* bias, int bias_dtype,
                       int activation, void* stream, int variant) {
    Epilogue ep;
    ep.bias = bias;
    ep.bias_kind = bias_dtype;
    ep.act = activation;
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant, kWsInternal, nullptr, 0,
                    ep);
}

int gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
             int64_t ldc, float alpha, float beta, int out_dtype, int in_format, void* stream, int variant) {
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant, kWsInternal, nullptr, 0,
                    Epilogue(), 1, in_format);
}

int gemm_fp8_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_format, const void* B,
                int64_t ldb, int b_format, void* C, int64_t ldc, float alpha, float beta, int out_dtype, void* stream,
                int variant, void* workspace, int64_t workspace_bytes) {
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant,
                    workspace ? kWsCaller : kWsInternal, workspace, workspace_bytes, Epilogue(), 1, a_format, false,
                    false, -1, 0, b_format);
}

int gemm_quant_i8(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                  int in_type, void* Q, int64_t ldq, float alpha, const void* bias, int bias_dtype, int activation,
                  const float* row_scale, int zero_point, void* stream, int variant) {
    if (in_type < TCGEMM_IN_BF16 || in_type > TCGEMM_IN_E5M2) {
        t_last_error[0] = '\0';
        set_error("unknown operand type %d", in_type);
        return TCGEMM_ERR_INVALID_ARG;
    }
    Epilogue ep;
    ep.bias = bias;
    ep.bias_kind = bias_dtype;
    ep.act = activation;
    ep.qscale = row_scale;
    ep.qzero = zero_point;
    const int in_kind = in_type == TCGEMM_IN_BF16 ? 0 : 1;
    const int in_fmt = in_type == TCGEMM_IN_E5M2 ? TCGEMM_FP8_E5M2 : TCGEMM_FP8_E4M3;
    return run_gemm(M, N, K, A, lda, B, ldb, Q, ldq, alpha, 0.0f, TCGEMM_OUT_I8, stream, variant, kWsInternal, nullptr,
                    0, ep, in_kind, in_fmt);
}

int gemm_bf16_layout(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_layout, const void* B,
                     int64_t ldb, int b_layout, void* C, int64_t ldc, float alpha, float beta, int out_dtype,
                     void* stream, int variant) {
    if ((a_layout != TCGEMM_ROW_MAJOR && a_layout != TCGEMM_COL_MAJOR) ||
        (b_layout != TCGEMM_ROW_MAJOR && b_layout != TCGEMM_COL_MAJOR)) {
        t_last_error[0] = '\0';
        set_error("layouts must be TCGEMM_ROW_MAJOR (0) or TCGEMM_COL_MAJOR (1)");
        return TCGEMM_ERR_INVALID_ARG;
    }
    return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant, kWsInternal, nullptr, 0,
                    Epilogue(), 0, 0, a_layout == TCGEMM_COL_MAJOR, b_layout == TCGEMM_ROW_MAJOR);
}

int tcgemm_autotune(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_layout, const void* B,
                    int64_t ldb, int b_layout, int in_type, void* C, int64_t ldc, float alpha, float beta,
                    int out_dtype, int iters, void* flush, int64_t flush_bytes, void* stream_v, int* best_variant,
                    float* best_us) {
    t_last_error[0] = '\0';
    if (best_variant == nullptr || iters <= 0 || iters > 1000 || in_type < TCGEMM_IN_BF16 ||
        in_type > TCGEMM_IN_E5M2 || (out_dtype != TCGEMM_OUT_F32 && out_dtype != TCGEMM_OUT_BF16) ||
        (a_layout != TCGEMM_ROW_MAJOR && a_layout != TCGEMM_COL_MAJOR) ||
        (b_layout != TCGEMM_ROW_MAJOR && b_layout != TCGEMM_COL_MAJOR) || M <= 0 || N <= 0 || K <= 0 ||
        flush_bytes < 0 || (flush_bytes > 0 && flush == nullptr)) {
        set_error("autotune: bad arguments (sizes > 0, 1 <= iters <= 1000, fp32 or bf16 output)");
        return TCGEMM_ERR_INVALID_ARG;
    }
    const int in_kind = in_type == TCGEMM_IN_BF16 ? 0 : 1;
    const int in_fmt = in_type == TCGEMM_IN_E5M2 ? TCGEMM_FP8_E5M2 : TCGEMM_FP8_E4M3;
    const bool a_col = a_layout == TCGEMM_COL_MAJOR, b_row = b_layout == TCGEMM_ROW_MAJOR;
    int dev = 0;
    DeviceInfo info;
    int rc = probe_device(dev, info);
    if (rc != TCGEMM_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    auto call = [&](int v) {
        return run_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream_v, v, kWsInternal, nullptr, 0,
                        Epilogue(), in_kind, in_fmt, a_col, b_row);
    };
    // One event pair per timed call: with a flush buffer, each call is timed
    // alone after the buffer (larger than L2) has been written, so the
    // operands come from memory as in a cold call.
    std::vector<cudaEvent_t> ev(2 * static_cast<size_t>(iters), nullptr);
    for (auto& e : ev) {
        if (cudaEventCreate(&e) != cudaSuccess) {
            for (auto& f : ev)
                if (f) cudaEventDestroy(f);
            set_error("autotune: cudaEventCreate failed");
            return TCGEMM_ERR_CUDA;
        }
    }
    const int candidates[] = {TCGEMM_VARIANT_2CTA,      TCGEMM_VARIANT_2CTA_W256,    TCGEMM_VARIANT_1CTA,
                              TCGEMM_VARIANT_1CTA_N64,  TCGEMM_VARIANT_SWAP_N64,     TCGEMM_VARIANT_SWAP_N64_KS2,
                              TCGEMM_VARIANT_SWAP_PAIR};
    int best = TCGEMM_VARIANT_AUTO;
    float best_t = 0.0f;
    rc = TCGEMM_OK;
    for (int v : candidates) {
        if (call(v) != TCGEMM_OK) continue;  // not built for these operands / layouts
        bool ok = true;
        for (int i = 0; i < iters && ok; ++i) {
            if (flush_bytes > 0 && cudaMemsetAsync(flush, i & 0xFF, static_cast<size_t>(flush_bytes), stream) !=
                                       cudaSuccess) {
                ok = false;
                break;
            }
            ok = cudaEventRecord(ev[2 * i], stream) == cudaSuccess && call(v) == TCGEMM_OK &&
                 cudaEventRecord(ev[2 * i + 1], stream) == cudaSuccess;
        }
        if (!ok || cudaEventSynchronize(ev.back()) != cudaSuccess) {
            rc = TCGEMM_ERR_CUDA;
            break;
        }
        float total_ms = 0.0f;
        for (int i = 0; i < iters; ++i) {
            float ms = 0.0f;
            cudaEventElapsedTime(&ms, ev[2 * i], ev[2 * i + 1]);
            total_ms += ms;
        }
        const float us = total_ms * 1000.0f / static_cast<float>(iters);
        if (best == TCGEMM_VARIANT_AUTO || us < best_t) {
            best = v;
            best_t = us;
        }
    }
    for (auto& e : ev) cudaEventDestroy(e);
    if (rc != TCGEMM_OK) {
        set_error("autotune: a timed call failed");
        return rc;
    }
    if (best == TCGEMM_VARIANT_AUTO) {
        set_error("autotune: no variant ran for this problem");
        return TCGEMM_ERR_INVALID_ARG;
    }
    // The device status word records any timeout of the runs above.
    uint32_t where = 0;
    rc = tcgemm_check_device_status(stream_v, &where);
    if (rc != TCGEMM_OK) return rc;
    {
        std::lock_guard<std::mutex> lk(g_tune_mu);
        g_tuned[TuneKey{dev, M, N, K, in_kind, in_kind == 1 ? in_fmt : 0, out_dtype, a_col ? 1 : 0, b_row ? 1 : 0,
                        beta != 0.0f ? 1 : 0}] = best;
    }
    *best_variant = best;
    if (best_us) *best_us = best_t;
    return TCGEMM_OK;
}

int tcgemm_autotune_lookup(int64_t M, int64_t N, int64_t K, int in_type, int out_dtype, int a_layout, int b_layout,
                           int beta_nonzero) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        dev = 0;
    }
    const int in_kind = in_type == TCGEMM_IN_BF16 ? 0 : 1;
    const int in_fmt = in_type == TCGEMM_IN_E5M2 ? TCGEMM_FP8_E5M2 : TCGEMM_FP8_E4M3;
    return tuned_variant(TuneKey{dev, M, N, K, in_kind, in_kind == 1 ? in_fmt : 0, out_dtype,
                                 a_layout == TCGEMM_COL_MAJOR ? 1 : 0, b_layout == TCGEMM_ROW_MAJOR ? 1 : 0,
                                 beta_nonzero ? 1 : 0});
}

void tcgemm_autotune_clear(void) {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    g_tuned.clear();
}

int64_t tcgemm_noalloc_scratch_bytes(void) { return static_cast<int64_t>(kNoAllocScratchBytes); }

int tcgemm_noalloc_fits(int64_t M, int64_t N, int64_t K, int variant, int num_sms) {
    if (M <= 0 || N <= 0 || K <= 0 || num_sms <= 0 || !variant_known(variant)) return -1;
    Plan pl;
    if (!make_plan(M, N, K, variant, num_sms, num_sms / 2, pl)) return -1;
    return noalloc_fits(pl.ws_bytes) ? 1 : 0;
}

int64_t tcgemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int variant, int num_sms) {
    if (M <= 0 || N <= 0 || K <= 0 || num_sms <= 0) return 0;
    Plan pl;
    if (!make_plan(M, N, K, variant, num_sms, num_sms / 2, pl)) return -1;
    return static_cast<int64_t>(pl.ws_bytes);
}

int tcgemm_pick_variant(int64_t M, int64_t N, int64_t K, int num_sms) { return pick_variant(M, N, K, num_sms); }

int tcgemm_plan(int64_t M, int64_t N, int64_t K, int variant, int num_sms, int64_t* out) {
    if (out == nullptr || M <= 0 || N <= 0 || K <= 0 || num_sms <= 0) return TCGEMM_ERR_INVALID_ARG;
    Plan pl;
    if (!make_plan(M, N, K, variant, num_sms, num_sms / 2, pl)) return TCGEMM_ERR_INVALID_ARG;
    fill_plan_out(pl, out);
    return TCGEMM_OK;
}

int tcgemm_plan_kind(int64_t M, int64_t N, int64_t K, int variant, int in_kind, int a_layout, int b_layout,
                     int num_sms, int64_t* out) {
    if (out == nullptr || M <= 0 || N <= 0 || K <= 0 || num_sms <= 0 || in_kind < 0 || in_kind > 1)
        return TCGEMM_ERR_INVALID_ARG;
    Plan pl;
    if (!make_plan(M, N, K, variant, num_sms, num_sms / 2, pl, true, in_kind,
                   a_layout == TCGEMM_COL_MAJOR, b_layout == TCGEMM_ROW_MAJOR))
        return TCGEMM_ERR_INVALID_ARG;
    fill_plan_out(pl, out);
    return TCGEMM_OK;
}

int tcgemm_device_info(int64_t* out) {
    if (out == nullptr) return TCGEMM_ERR_INVALID_ARG;
    int dev = 0;
    DeviceInfo info;
    const int rc = probe_device(dev, info);
    if (rc != TCGEMM_OK) return rc;
    out[0] = info.sms;
    out[1] = info.max_pairs;
    out[2] = 0;  // formerly the 4-CTA cluster count; no 4-CTA kernel is built
    out[3] = dev;
    return TCGEMM_OK;
}

int tcgemm_plan_device(int64_t M, int64_t N, int64_t K, int variant, int64_t* out) {
    int64_t d[4];
    const int rc = tcgemm_device_info(d);
    if (rc != TCGEMM_OK) return rc;
    if (out == nullptr || M <= 0 || N <= 0 || K <= 0) return TCGEMM_ERR_INVALID_ARG;
    Plan pl;
    if (!make_plan(M, N, K, variant, static_cast<int>(d[0]), static_cast<int>(d[1]), pl))
        return TCGEMM_ERR_INVALID_ARG;
    fill_plan_out(pl, out);
    return TCGEMM_OK;
}

int tcgemm_units(int64_t M, int64_t N, int64_t K, int variant, int num_sms, int cluster, int max_units,
                 int32_t* out) {
    if (out == nullptr || M <= 0 || N <= 0 || K <= 0 || num_sms <= 0 || max_units < 0) return -1;
    Plan pl;
    if (!make_plan(M, N, K, variant, num_sms, num_sms / 2, pl)) return -1;
    const int clusters = pl.grid / (pl.cta_group * pl.ks);
    if (cluster < 0 || cluster >= clusters) return -1;
    tcg::GemmParams gp = {};
    gp.num_kb = pl.num_kb;
    gp.tiles_dp = pl.tiles_dp;
    gp.sk_tiles = pl.sk_tiles;
    gp.sk_iters = pl.sk_iters;
    tcg::UnitIter it(cluster, clusters);
    it.start(gp);
    tcg::WorkUnit u;
    int n = 0;
    while (it.next(gp, u)) {
        if (n < max_units) {
            int32_t* o = out + 7 * n;
            o[0] = u.tile;
            o[1] = u.kb0;
            o[2] = u.kb1;
            o[3] = u.slot;
            o[4] = u.sk_tile;
            o[5] = u.piece;
            o[6] = u.npieces;
        }
        ++n;
    }
    return n;
}

int tcgemm_tile_order_hilbert(int tiles_m, int tiles_n, int64_t count, int32_t* tm, int32_t* tn) {
    if (tiles_m <= 0 || tiles_n <= 0 || count < 0 || count > static_cast<int64_t>(tiles_m) * tiles_n ||
        tm == nullptr || tn == nullptr)
        return TCGEMM_ERR_INVALID_ARG;
    int k = 0;
    while ((1 << k) < std::max(tiles_m, tiles_n)) ++k;
    for (int64_t t = 0; t < count; ++t) {
        int a, b;
        tcg::hilbert_tile(static_cast<int>(t), tiles_m, tiles_n, k, a, b);
        tm[t] = a;
        tn[t] = b;
    }
    return TCGEMM_OK;
}

int tcgemm_tile_order(int tiles_m, int tiles_n, int group_m, int64_t count, int32_t* tm, int32_t* tn) {
    if (tiles_m <= 0 || tiles_n <= 0 || group_m <= 0 || count < 0 || tm == nullptr || tn == nullptr)
        return TCGEMM_ERR_INVALID_ARG;
    for (int64_t t = 0; t < count; ++t) {
        int a, b;
        tcg::grouped_tile(static_cast<int>(t), tiles_m, tiles_n, group_m, a, b);
        tm[t] = a;
        tn[t] = b;
    }
    return TCGEMM_OK;
}

const char* tcgemm_status_string(int status) {
    switch (status) {
        case TCGEMM_OK: return "TCGEMM_OK";
        case TCGEMM_ERR_INVALID_ARG: return "TCGEMM_ERR_INVALID_ARG";
        case TCGEMM_ERR_ALIGNMENT: return "TCGEMM_ERR_ALIGNMENT";
        case TCGEMM_ERR_UNSUPPORTED_DEVICE: return "TCGEMM_ERR_UNSUPPORTED_DEVICE";
        case TCGEMM_ERR_CUDA: return "TCGEMM_ERR_CUDA";
        case TCGEMM_ERR_TIMEOUT: return "TCGEMM_ERR_TIMEOUT";
        default: return "TCGEMM_ERR_UNKNOWN";
    }
}

const char* tcgemm_last_error(void) { return t_last_error; }

int tcgemm_check_device_status(void* stream, uint32_t* where_out) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_error("cudaStreamSynchronize: %s", cudaGetErrorString(e));
        return TCGEMM_ERR_CUDA;
    }
    uint32_t st[4] = {0, 0, 0, 0};
    e = cudaMemcpyFromSymbol(st, tcg::g_tcgemm_status, sizeof st);
    if (e != cudaSuccess) {
        set_error("reading the status word: %s", cudaGetErrorString(e));
        return TCGEMM_ERR_CUDA;
    }
    if (st[0] == 0) return TCGEMM_OK;
    const uint32_t zero[4] = {0, 0, 0, 0};
    e = cudaMemcpyToSymbol(tcg::g_tcgemm_status, zero, sizeof zero);
    if (where_out) *where_out = st[1];
    set_error("device wait timed out (role %u, block %u)", st[1], st[2]);
    if (e != cudaSuccess) return TCGEMM_ERR_CUDA;
    return st[0] == tcg::kStatusTimeout ? TCGEMM_ERR_TIMEOUT : TCGEMM_ERR_CUDA;
}

int tcgemm_selftest_timeout(void* stream, uint64_t timeout_ns_arg) {
    int dev = 0;
    DeviceInfo info;
    int rc = probe_device(dev, info);
    if (rc != TCGEMM_OK) return rc;
    if (timeout_ns_arg == 0 || timeout_ns_arg > 10ull * 1000 * 1000 * 1000) {
        set_error("self-test timeout must be in (0, 10 s]");
        return TCGEMM_ERR_INVALID_ARG;
    }
    tcg::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns_arg);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kernel launch: %s", cudaGetErrorString(e));
        return TCGEMM_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return tcgemm_check_device_status(stream, nullptr);
}

int tcgemm_selftest_withheld_load(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                  int64_t ldb, void* C, int64_t ldc, int variant, uint64_t timeout_ns_arg,
                                  void* stream) {
    t_last_error[0] = '\0';
    if (variant != TCGEMM_VARIANT_1CTA && variant != TCGEMM_VARIANT_2CTA && variant != TCGEMM_VARIANT_1CTA_N64 &&
        variant != TCGEMM_VARIANT_2CTA_W256) {
        set_error("the withheld-load self test runs the plain-product variants 1, 2, 4 and 5");
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (M <= 0 || N <= 0 || K <= 0 || timeout_ns_arg == 0 || timeout_ns_arg > 10ull * 1000 * 1000 * 1000) {
        set_error("self test: sizes must be positive and the limit in (0, 10 s]");
        return TCGEMM_ERR_INVALID_ARG;
    }
    // No split: the withheld k-block is the first one CTA 0 loads, in a whole tile.
    const int rc = run_gemm(M, N, K, A, lda, B, ldb, C, ldc, 1.0f, 0.0f, TCGEMM_OUT_F32, stream, variant, kWsNone,
                            nullptr, 0, Epilogue(), 0, 0, false, false, 0, timeout_ns_arg);
    if (rc != TCGEMM_OK) return rc;
    return tcgemm_check_device_status(stream, nullptr);
}

uint64_t tcgemm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int tcgemm_version(void) { return 100; }

}  // extern "C"

// The host-buffer entry point (gemm_bf16_host) and its device copies.
#include "host_entry.cuh"

// Saving, loading and setting the tuned-choice table.
#include "tune_table.cuh"
