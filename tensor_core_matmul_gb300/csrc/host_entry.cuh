// The C ABI's host-buffer entry points: gemm_bf16_host and gemm_fp8_host copy
// A, B (and C when beta != 0) from host memory to the library's device copies,
// run the GEMM there and copy C back, all on the caller's stream.  Included once,
// at the end of tcgemm.cu (it uses that file's validation, device probe and
// launch path).
#pragma once

namespace {

// Device copies of the operands and of C for gemm_bf16_host, one set per
// (device, stream) so that calls on different streams never share them.
// Grown (never shrunk) when a call needs more; cudaFree waits for the device,
// so a buffer is never freed under a copy or kernel still using it.
struct HostStage {
    void* p[3] = {nullptr, nullptr, nullptr};  // A, B, C
    uint64_t bytes[3] = {0, 0, 0};
};
std::mutex g_stage_mu;
std::map<std::pair<int, uintptr_t>, HostStage> g_stage;

int host_stage(int dev, cudaStream_t stream, const uint64_t need[3], void* out[3]) {
    std::lock_guard<std::mutex> lk(g_stage_mu);
    HostStage& st = g_stage[{dev, reinterpret_cast<uintptr_t>(stream)}];
    for (int i = 0; i < 3; ++i) {
        if (need[i] > st.bytes[i]) {
            const uint64_t grain = uint64_t{2} << 20;
            const uint64_t bytes = (need[i] + grain - 1) / grain * grain;
            if (st.p[i]) {
                cudaFree(st.p[i]);
                st.p[i] = nullptr;
                st.bytes[i] = 0;
            }
            cudaError_t e = cudaMalloc(&st.p[i], bytes);
            if (e != cudaSuccess) {
                st.p[i] = nullptr;
                set_error("staging cudaMalloc(%llu): %s", static_cast<unsigned long long>(bytes),
                          cudaGetErrorString(e));
                return TCGEMM_ERR_CUDA;
            }
            st.bytes[i] = bytes;
        }
        out[i] = st.p[i];
    }
    return TCGEMM_OK;
}

// `rows` rows of `width` bytes, `pitch` bytes apart on both sides: one plain
// copy when the rows are contiguous, else one pitched copy (which leaves the
// padding between rows alone).
cudaError_t copy_matrix(void* dst, const void* src, int64_t pitch, int64_t width, int64_t rows, cudaMemcpyKind kind,
                        cudaStream_t s) {
    if (pitch == width) return cudaMemcpyAsync(dst, src, static_cast<size_t>(width * rows), kind, s);
    return cudaMemcpy2DAsync(dst, static_cast<size_t>(pitch), src, static_cast<size_t>(pitch),
                             static_cast<size_t>(width), static_cast<size_t>(rows), kind, s);
}

// in_kind 0: bf16 operands; 1: 8-bit operands in format in_fmt (both).
int host_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
              int64_t ldc, float alpha, float beta, int out_dtype, void* stream, int in_kind, int in_fmt) {
    t_last_error[0] = '\0';
    if (out_dtype != TCGEMM_OUT_F32 && out_dtype != TCGEMM_OUT_BF16) {
        set_error("out_dtype must be TCGEMM_OUT_F32 (0) or TCGEMM_OUT_BF16 (1), got %d", out_dtype);
        return TCGEMM_ERR_INVALID_ARG;
    }
    if (in_kind == 1 && in_fmt != TCGEMM_FP8_E4M3 && in_fmt != TCGEMM_FP8_E5M2) {
        set_error("unknown FP8 format %d", in_fmt);
        return TCGEMM_ERR_INVALID_ARG;
    }
    const int64_t isz = in_kind == 1 ? 1 : 2;  // bytes per operand element
    // The host buffers follow the device entry points' rules (sizes, leading
    // dimensions, 16-byte alignment, no overlap of C with A or B).
    int rc = validate(M, N, K, A, lda, B, ldb, C, ldc, out_dtype, isz);
    if (rc != TCGEMM_OK) return rc;
    if (M == 0 || N == 0) return TCGEMM_OK;
    int dev = 0;
    DeviceInfo info;
    rc = probe_device(dev, info);
    if (rc != TCGEMM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint64_t esz = out_dtype == TCGEMM_OUT_F32 ? 4 : 2;
    const uint64_t need[3] = {K > 0 ? static_cast<uint64_t>(((M - 1) * lda + K) * isz) : 0,
                              K > 0 ? static_cast<uint64_t>(((N - 1) * ldb + K) * isz) : 0,
                              static_cast<uint64_t>((N - 1) * ldc + M) * esz};
    void* d[3] = {nullptr, nullptr, nullptr};
    rc = host_stage(dev, s, need, d);
    if (rc != TCGEMM_OK) return rc;
    // One copy per matrix, all on the caller's stream: only the matrices' own
    // elements move (the device copies keep the caller's leading dimensions),
    // so C's padding on the host is never written.
    cudaError_t e = cudaSuccess;
    if (K > 0) {
        e = copy_matrix(d[0], A, lda * isz, K * isz, M, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = copy_matrix(d[1], B, ldb * isz, K * isz, N, cudaMemcpyHostToDevice, s);
    }
    if (e == cudaSuccess && beta != 0.0f) e = copy_matrix(d[2], C, ldc * esz, M * esz, N, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) {
        set_error("host-to-device copy: %s", cudaGetErrorString(e));
        return TCGEMM_ERR_CUDA;
    }
    rc = run_gemm(M, N, K, d[0], lda, d[1], ldb, d[2], ldc, alpha, beta, out_dtype, stream, TCGEMM_VARIANT_AUTO,
                  kWsInternal, nullptr, 0, Epilogue(), in_kind, in_fmt);
    if (rc != TCGEMM_OK) return rc;
    e = copy_matrix(C, d[2], ldc * esz, M * esz, N, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) {
        set_error("device-to-host copy: %s", cudaGetErrorString(e));
        return TCGEMM_ERR_CUDA;
    }
    return TCGEMM_OK;
}

}  // namespace

extern "C" {

int gemm_bf16_host(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                   void* C, int64_t ldc, float alpha, float beta, int out_dtype, void* stream) {
    return host_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, 0, 0);
}

int gemm_fp8_host(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                  void* C, int64_t ldc, float alpha, float beta, int out_dtype, int in_format, void* stream) {
    return host_gemm(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, 1, in_format);
}

}  // extern "C"
