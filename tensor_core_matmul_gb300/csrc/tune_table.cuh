// The tuned-choice table's persistence: record a choice by hand, write the
// table to a text file and read it back, so that a process can start with
// the choices tcgemm_autotune made in an earlier one.  Included once, at the
// end of tcgemm.cu (it uses that file's table, key and error state).
#pragma once

#include <cstdio>
#include <vector>

namespace {

constexpr const char* kTuneFileHeader = "tcgemm-autotune 1";

int current_device_or_zero() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        dev = 0;
    }
    return dev;
}

// Whether `variant` is built for this kind of problem (what tcgemm_autotune
// could have chosen).
bool tune_entry_valid(const TuneKey& k, int variant) {
    const int64_t lim = (int64_t{1} << 31) - 1;
    if (k.dev < 0 || k.dev >= kMaxDevices || k.M < 1 || k.N < 1 || k.K < 1 || k.M > lim || k.N > lim || k.K > lim)
        return false;
    if (k.in_kind != 0 && k.in_kind != 1) return false;
    if (k.in_kind == 0 && k.in_fmt != 0) return false;
    if (k.in_kind == 1 && k.in_fmt != TCGEMM_FP8_E4M3 && k.in_fmt != TCGEMM_FP8_E5M2) return false;
    if (k.out_dtype != TCGEMM_OUT_F32 && k.out_dtype != TCGEMM_OUT_BF16 && k.out_dtype != TCGEMM_OUT_I8) return false;
    if ((k.a_col | k.b_row | k.has_beta) & ~1) return false;
    if (!variant_known(variant) || variant == TCGEMM_VARIANT_AUTO) return false;
    if (variant == TCGEMM_VARIANT_1CTA && (k.in_kind == 1 || k.out_dtype == TCGEMM_OUT_I8)) return false;
    if (variant == TCGEMM_VARIANT_SWAP_PAIR &&
        (k.in_kind == 1 || k.out_dtype == TCGEMM_OUT_I8 || k.a_col || k.b_row || k.M > 128))
        return false;
    if ((k.a_col || k.b_row) && k.in_kind == 1) return false;
    if (k.out_dtype == TCGEMM_OUT_I8 && k.has_beta) return false;
    return true;
}

}  // namespace

extern "C" {

int tcgemm_autotune_set(int64_t M, int64_t N, int64_t K, int in_type, int out_dtype, int a_layout, int b_layout,
                        int beta_nonzero, int variant) {
    t_last_error[0] = '\0';
    if (in_type != TCGEMM_IN_BF16 && in_type != TCGEMM_IN_E4M3 && in_type != TCGEMM_IN_E5M2) {
        set_error("unknown in_type %d", in_type);
        return TCGEMM_ERR_INVALID_ARG;
    }
    const int in_kind = in_type == TCGEMM_IN_BF16 ? 0 : 1;
    const int in_fmt = in_kind == 0 ? 0 : (in_type == TCGEMM_IN_E5M2 ? TCGEMM_FP8_E5M2 : TCGEMM_FP8_E4M3);
    const TuneKey key{current_device_or_zero(), M, N, K, in_kind, in_fmt, out_dtype,
                      a_layout == TCGEMM_COL_MAJOR ? 1 : 0, b_layout == TCGEMM_ROW_MAJOR ? 1 : 0,
                      beta_nonzero ? 1 : 0};
    if (variant == TCGEMM_VARIANT_AUTO) {
        std::lock_guard<std::mutex> lk(g_tune_mu);
        g_tuned.erase(key);
        return TCGEMM_OK;
    }
    if (!tune_entry_valid(key, variant)) {
        set_error("variant %d is not built for this problem (or a size or type is out of range)", variant);
        return TCGEMM_ERR_INVALID_ARG;
    }
    std::lock_guard<std::mutex> lk(g_tune_mu);
    g_tuned[key] = variant;
    return TCGEMM_OK;
}

int64_t tcgemm_autotune_save(const char* path) {
    t_last_error[0] = '\0';
    if (path == nullptr) {
        set_error("null path");
        return -1;
    }
    std::vector<std::pair<TuneKey, int>> rows;
    {
        std::lock_guard<std::mutex> lk(g_tune_mu);
        rows.assign(g_tuned.begin(), g_tuned.end());
    }
    FILE* f = std::fopen(path, "w");
    if (!f) {
        set_error("cannot open %s for writing", path);
        return -1;
    }
    bool ok = std::fprintf(f, "%s\n", kTuneFileHeader) > 0;
    for (const auto& r : rows) {
        const TuneKey& k = r.first;
        ok = ok && std::fprintf(f, "%d %lld %lld %lld %d %d %d %d %d %d %d\n", k.dev, static_cast<long long>(k.M),
                                static_cast<long long>(k.N), static_cast<long long>(k.K), k.in_kind, k.in_fmt,
                                k.out_dtype, k.a_col, k.b_row, k.has_beta, r.second) > 0;
    }
    ok = (std::fclose(f) == 0) && ok;
    if (!ok) {
        set_error("writing %s failed", path);
        return -1;
    }
    return static_cast<int64_t>(rows.size());
}

int64_t tcgemm_autotune_load(const char* path) {
    t_last_error[0] = '\0';
    if (path == nullptr) {
        set_error("null path");
        return -1;
    }
    FILE* f = std::fopen(path, "r");
    if (!f) {
        set_error("cannot open %s", path);
        return -1;
    }
    char line[256];
    std::vector<std::pair<TuneKey, int>> rows;
    bool ok = std::fgets(line, sizeof line, f) != nullptr &&
              std::strncmp(line, kTuneFileHeader, std::strlen(kTuneFileHeader)) == 0;
    if (!ok) set_error("%s: not a table written by tcgemm_autotune_save", path);
    int64_t lineno = 1;
    while (ok && std::fgets(line, sizeof line, f) != nullptr) {
        ++lineno;
        if (line[0] == '\n' || line[0] == '\0') continue;
        TuneKey k{};
        long long m = 0, n = 0, kk = 0;
        int variant = 0;
        char extra = 0;
        const int got = std::sscanf(line, "%d %lld %lld %lld %d %d %d %d %d %d %d %c", &k.dev, &m, &n, &kk,
                                    &k.in_kind, &k.in_fmt, &k.out_dtype, &k.a_col, &k.b_row, &k.has_beta, &variant,
                                    &extra);
        k.M = m;
        k.N = n;
        k.K = kk;
        if (got != 11 || !tune_entry_valid(k, variant)) {
            set_error("%s line %lld: not a tuned choice", path, static_cast<long long>(lineno));
            ok = false;
            break;
        }
        rows.emplace_back(k, variant);
    }
    std::fclose(f);
    if (!ok) return -1;
    std::lock_guard<std::mutex> lk(g_tune_mu);
    for (const auto& r : rows) g_tuned[r.first] = r.second;
    return static_cast<int64_t>(rows.size());
}

}  // extern "C"
