"""ctypes binding of the tcgemm C ABI (include/tcgemm.h).

Argument marshalling only: every step of the GEMM runs in the CUDA library.
There is no fallback: if libtcgemm.so is missing or fails to load, every call
raises.  Torch is used for device memory and streams.

Storage convention for torch tensors (matching the C ABI's layouts):
  A: (M, lda) bf16       -> A[i, k]   (row-major M x K)
  B: (N, ldb) bf16       -> B[k, j] is B_t[j, k] (column-major K x N)
  C: (N, ldc) fp32/bf16  -> C[i, j] is C_t[j, i] (column-major M x N)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

OUT_F32 = 0
OUT_BF16 = 1
OUT_I8 = 2
IN_BF16, IN_E4M3, IN_E5M2 = range(3)
ROW_MAJOR, COL_MAJOR = range(2)
VARIANT_AUTO, VARIANT_1CTA, VARIANT_2CTA = 0, 1, 2        # 3 names no kernel
VARIANT_1CTA_N64, VARIANT_2CTA_W256, VARIANT_SWAP_N64, VARIANT_SWAP_N64_KS2 = 4, 5, 6, 7

ACT_NONE, ACT_RELU, ACT_GELU, ACT_GELU_TANH = range(4)
ACTIVATIONS = {"none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU, "gelu_tanh": ACT_GELU_TANH}
BIAS_NONE, BIAS_F32, BIAS_BF16 = range(3)
FP8_E4M3, FP8_E5M2 = range(2)
FP8_FORMATS = {"e4m3": FP8_E4M3, "e5m2": FP8_E5M2}

STATUS = {0: "TCGEMM_OK", 1: "TCGEMM_ERR_INVALID_ARG", 2: "TCGEMM_ERR_ALIGNMENT",
          3: "TCGEMM_ERR_UNSUPPORTED_DEVICE", 4: "TCGEMM_ERR_CUDA", 5: "TCGEMM_ERR_TIMEOUT"}


class TcgemmError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {detail}")


_lib = None


def lib_path() -> str:
    return os.environ.get("TCGEMM_LIB", _build.LIB_PATH)


def lib() -> ctypes.CDLL:
    """Load libtcgemm.so (built in-tree by __graft_entry__.build() or
    tensor_core_matmul_gb300._build.build()).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libtcgemm.so not found at {path}; build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    i64, p, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    gemm_args = [i64, i64, i64, p, i64, p, i64, p, i64, f32, f32, i32, p]
    L.gemm_bf16.argtypes = gemm_args
    L.gemm_bf16.restype = i32
    L.gemm_bf16_variant.argtypes = gemm_args + [i32]
    L.gemm_bf16_variant.restype = i32
    L.gemm_bf16_ws.argtypes = gemm_args + [i32, p, i64]
    L.gemm_bf16_ws.restype = i32
    L.gemm_bf16_bias_act.argtypes = gemm_args[:-1] + [p, i32, i32, p, i32]
    L.gemm_bf16_bias_act.restype = i32
    L.gemm_quant_i8.argtypes = [i64, i64, i64, p, i64, p, i64, i32, p, i64, f32, p, i32, i32, p, i32, p, i32]
    L.gemm_quant_i8.restype = i32
    L.gemm_bf16_layout.argtypes = [i64, i64, i64, p, i64, i32, p, i64, i32, p, i64, f32, f32, i32, p, i32]
    L.gemm_bf16_layout.restype = i32
    L.tcgemm_autotune.argtypes = [i64, i64, i64, p, i64, i32, p, i64, i32, i32, p, i64, f32, f32, i32, i32, p, i64,
                                  p, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float)]
    L.tcgemm_autotune.restype = i32
    L.tcgemm_autotune_lookup.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32]
    L.tcgemm_autotune_lookup.restype = i32
    L.tcgemm_autotune_clear.argtypes = []
    L.tcgemm_autotune_clear.restype = None
    L.tcgemm_autotune_set.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32]
    L.tcgemm_autotune_set.restype = i32
    L.tcgemm_autotune_save.argtypes = [ctypes.c_char_p]
    L.tcgemm_autotune_save.restype = i64
    L.tcgemm_autotune_load.argtypes = [ctypes.c_char_p]
    L.tcgemm_autotune_load.restype = i64
    L.gemm_fp8.argtypes = gemm_args[:-1] + [i32, p, i32]
    L.gemm_fp8.restype = i32
    L.gemm_fp8_ex.argtypes = [i64, i64, i64, p, i64, i32, p, i64, i32, p, i64, f32, f32, i32, p, i32, p, i64]
    L.gemm_fp8_ex.restype = i32
    L.gemm_fp8_host.argtypes = gemm_args[:-1] + [i32, p]
    L.gemm_fp8_host.restype = i32
    L.tcgemm_plan_kind.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int64)]
    L.tcgemm_plan_kind.restype = i32
    L.gemm_bf16_noalloc.argtypes = gemm_args + [i32]
    L.gemm_bf16_noalloc.restype = i32
    L.gemm_bf16_host.argtypes = gemm_args
    L.gemm_bf16_host.restype = i32
    L.tcgemm_noalloc_scratch_bytes.argtypes = []
    L.tcgemm_noalloc_scratch_bytes.restype = i64
    L.tcgemm_noalloc_fits.argtypes = [i64, i64, i64, i32, i32]
    L.tcgemm_noalloc_fits.restype = i32
    L.tcgemm_workspace_bytes.argtypes = [i64, i64, i64, i32, i32]
    L.tcgemm_workspace_bytes.restype = i64
    L.tcgemm_pick_variant.argtypes = [i64, i64, i64, i32]
    L.tcgemm_pick_variant.restype = i32
    L.tcgemm_plan.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(ctypes.c_int64)]
    L.tcgemm_plan.restype = i32
    L.tcgemm_plan_device.argtypes = [i64, i64, i64, i32, ctypes.POINTER(ctypes.c_int64)]
    L.tcgemm_plan_device.restype = i32
    L.tcgemm_device_info.argtypes = [ctypes.POINTER(ctypes.c_int64)]
    L.tcgemm_device_info.restype = i32
    L.tcgemm_units.argtypes = [i64, i64, i64, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int32)]
    L.tcgemm_units.restype = i32
    L.tcgemm_tile_order.argtypes = [i32, i32, i32, i64, ctypes.POINTER(ctypes.c_int32),
                                    ctypes.POINTER(ctypes.c_int32)]
    L.tcgemm_tile_order.restype = i32
    L.tcgemm_tile_order_hilbert.argtypes = [i32, i32, i64, ctypes.POINTER(ctypes.c_int32),
                                            ctypes.POINTER(ctypes.c_int32)]
    L.tcgemm_tile_order_hilbert.restype = i32
    L.tcgemm_status_string.argtypes = [i32]
    L.tcgemm_status_string.restype = ctypes.c_char_p
    L.tcgemm_last_error.argtypes = []
    L.tcgemm_last_error.restype = ctypes.c_char_p
    L.tcgemm_check_device_status.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
    L.tcgemm_check_device_status.restype = i32
    L.tcgemm_selftest_timeout.argtypes = [p, ctypes.c_uint64]
    L.tcgemm_selftest_timeout.restype = i32
    L.tcgemm_selftest_withheld_load.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, i32, ctypes.c_uint64, p]
    L.tcgemm_selftest_withheld_load.restype = i32
    L.tcgemm_launch_count.argtypes = []
    L.tcgemm_launch_count.restype = ctypes.c_uint64
    L.tcgemm_version.argtypes = []
    L.tcgemm_version.restype = i32
    _lib = L
    return L


def last_error() -> str:
    return lib().tcgemm_last_error().decode(errors="replace")


def _check(status: int) -> None:
    if status != 0:
        raise TcgemmError(status, last_error())


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gemm_bf16_raw(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                  alpha: float, beta: float, out_dtype: int, stream: int, variant: int = 0) -> int:
    """Pointer-level call; returns the status code (no exception)."""
    L = lib()
    if variant == 0:
        return L.gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream)
    return L.gemm_bf16_variant(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant)


def gemm_bf16(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, M: Optional[int] = None,
              N: Optional[int] = None, K: Optional[int] = None, stream=None, variant: int = 0):
    """C = alpha * A * B + beta * C on the GPU, tensors in the storage
    convention above.  M, N, K default to C.shape[1], C.shape[0], A.shape[1]."""
    import torch
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("A, B and C must be CUDA tensors")
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise ValueError("A and B must be bfloat16")
    if C.dtype == torch.float32:
        out = OUT_F32
    elif C.dtype == torch.bfloat16:
        out = OUT_BF16
    else:
        raise ValueError("C must be float32 or bfloat16")
    for t in (A, B, C):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("A, B, C must be 2-D with unit inner stride")
    M = C.shape[1] if M is None else M
    N = C.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    if C.shape[0] < N or (K > 0 and (A.shape[0] < M or B.shape[0] < N)):
        raise ValueError("tensor shapes smaller than M/N")  # A and B are not read when K == 0
    st = gemm_bf16_raw(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(),
                       C.stride(0), float(alpha), float(beta), out, _stream_ptr(stream), variant)
    _check(st)
    return C


def gemm_bf16_host_raw(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                       alpha: float, beta: float, out_dtype: int, stream: int) -> int:
    """Pointer-level call of the host-buffer entry point; returns the status."""
    return lib().gemm_bf16_host(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream)


def gemm_bf16_host(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, M: Optional[int] = None,
                   N: Optional[int] = None, K: Optional[int] = None, stream=None):
    """C = alpha * A * B + beta * C with A, B, C in host memory (CPU tensors,
    pinned for asynchronous copies): the library copies them to the device,
    runs the GEMM and copies C back, all enqueued on `stream`.  C is valid
    once the stream has completed that work."""
    import torch
    if A.is_cuda or B.is_cuda or C.is_cuda:
        raise ValueError("A, B and C must be CPU tensors")
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise ValueError("A and B must be bfloat16")
    if C.dtype == torch.float32:
        out = OUT_F32
    elif C.dtype == torch.bfloat16:
        out = OUT_BF16
    else:
        raise ValueError("C must be float32 or bfloat16")
    for t in (A, B, C):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("A, B, C must be 2-D with unit inner stride")
    M = C.shape[1] if M is None else M
    N = C.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    if C.shape[0] < N or (K > 0 and (A.shape[0] < M or B.shape[0] < N)):
        raise ValueError("tensor shapes smaller than M/N")
    st = gemm_bf16_host_raw(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(),
                            C.stride(0), float(alpha), float(beta), out, _stream_ptr(stream))
    _check(st)
    return C


def gemm_bf16_bias_act_raw(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                           alpha: float, beta: float, out_dtype: int, bias: Optional[int], bias_dtype: int,
                           activation: int, stream: int, variant: int = 0) -> int:
    """Pointer-level call of the fused-epilogue entry point; returns the status."""
    return lib().gemm_bf16_bias_act(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, bias, bias_dtype,
                                    activation, stream, variant)


def gemm_bf16_bias_act(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, bias=None, activation="none",
                       M: Optional[int] = None, N: Optional[int] = None, K: Optional[int] = None, stream=None,
                       variant: int = 0):
    """C = act(alpha * A * B + beta * C + bias[j]) on the GPU (the fused
    epilogue), tensors as in gemm_bf16; ``bias`` a 1-D fp32 or bf16 CUDA
    tensor of at least N values (or None); ``activation`` one of ACTIVATIONS."""
    import torch
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("A, B and C must be CUDA tensors")
    if C.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("C must be float32 or bfloat16")
    out = OUT_F32 if C.dtype == torch.float32 else OUT_BF16
    M = C.shape[1] if M is None else M
    N = C.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise ValueError("A and B must be bfloat16")
    for t in (A, B, C):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("A, B, C must be 2-D with unit inner stride")
    if C.shape[0] < N or (K > 0 and (A.shape[0] < M or B.shape[0] < N)):
        raise ValueError("tensor shapes smaller than M/N")  # A and B are not read when K == 0
    if bias is None:
        bptr, bkind = None, BIAS_NONE
    else:
        if not bias.is_cuda or bias.dim() != 1 or bias.stride(0) != 1 or bias.shape[0] < N:
            raise ValueError("bias must be a contiguous 1-D CUDA tensor of at least N values")
        if bias.dtype == torch.float32:
            bkind = BIAS_F32
        elif bias.dtype == torch.bfloat16:
            bkind = BIAS_BF16
        else:
            raise ValueError("bias must be float32 or bfloat16")
        bptr = bias.data_ptr()
    act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
    st = gemm_bf16_bias_act_raw(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(),
                                C.stride(0), float(alpha), float(beta), out, bptr, bkind, act, _stream_ptr(stream),
                                variant)
    _check(st)
    return C


def gemm_fp8_raw(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                 alpha: float, beta: float, out_dtype: int, in_format: int, stream: int, variant: int = 0) -> int:
    """Pointer-level call of the 8-bit-operand entry point; returns the status."""
    return lib().gemm_fp8(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, in_format, stream, variant)


def gemm_fp8(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, M: Optional[int] = None, N: Optional[int] = None,
             K: Optional[int] = None, stream=None, variant: int = 0):
    """C = alpha * A * B + beta * C with A, B torch float8_e4m3fn or
    float8_e5m2 CUDA tensors (both the same), in the storage convention of
    gemm_bf16 (A (M, lda), B (N, ldb)); C float32 or bfloat16."""
    import torch
    fmts = {torch.float8_e4m3fn: FP8_E4M3, torch.float8_e5m2: FP8_E5M2}
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("A, B and C must be CUDA tensors")
    if A.dtype not in fmts or B.dtype != A.dtype:
        raise ValueError("A and B must both be float8_e4m3fn or both float8_e5m2")
    if C.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("C must be float32 or bfloat16")
    for t in (A, B, C):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("A, B, C must be 2-D with unit inner stride")
    M = C.shape[1] if M is None else M
    N = C.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    if C.shape[0] < N or (K > 0 and (A.shape[0] < M or B.shape[0] < N)):
        raise ValueError("tensor shapes smaller than M/N")
    out = OUT_F32 if C.dtype == torch.float32 else OUT_BF16
    st = gemm_fp8_raw(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(), C.stride(0),
                      float(alpha), float(beta), out, fmts[A.dtype], _stream_ptr(stream), variant)
    _check(st)
    return C


def gemm_fp8_ex(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, M: Optional[int] = None,
                N: Optional[int] = None, K: Optional[int] = None, stream=None, variant: int = 0, workspace=None):
    """gemm_fp8 with A and B each in its own 8-bit format (float8_e4m3fn or
    float8_e5m2, which may differ) and an optional caller workspace (a CUDA
    tensor, or None for the library's own)."""
    import torch
    fmts = {torch.float8_e4m3fn: FP8_E4M3, torch.float8_e5m2: FP8_E5M2}
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("A, B and C must be CUDA tensors")
    if A.dtype not in fmts or B.dtype not in fmts:
        raise ValueError("A and B must be float8_e4m3fn or float8_e5m2")
    if C.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("C must be float32 or bfloat16")
    for t in (A, B, C):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("A, B, C must be 2-D with unit inner stride")
    M = C.shape[1] if M is None else M
    N = C.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    out = OUT_F32 if C.dtype == torch.float32 else OUT_BF16
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().gemm_fp8_ex(M, N, K, A.data_ptr(), A.stride(0), fmts[A.dtype], B.data_ptr(), B.stride(0),
                             fmts[B.dtype], C.data_ptr(), C.stride(0), float(alpha), float(beta), out,
                             _stream_ptr(stream), variant, ws_ptr, ws_bytes))
    return C


def gemm_fp8_host(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, M: Optional[int] = None,
                  N: Optional[int] = None, K: Optional[int] = None, stream=None):
    """The host-buffer entry point for 8-bit operands: A, B, C are CPU torch
    tensors (A, B float8_e4m3fn or both float8_e5m2; C float32 or
    bfloat16), pinned for asynchronous copies."""
    import torch
    fmts = {torch.float8_e4m3fn: FP8_E4M3, torch.float8_e5m2: FP8_E5M2}
    if A.is_cuda or B.is_cuda or C.is_cuda:
        raise ValueError("A, B and C must be host tensors")
    if A.dtype not in fmts or B.dtype != A.dtype:
        raise ValueError("A and B must both be float8_e4m3fn or both float8_e5m2")
    M = C.shape[1] if M is None else M
    N = C.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    out = OUT_F32 if C.dtype == torch.float32 else OUT_BF16
    _check(lib().gemm_fp8_host(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(),
                               C.stride(0), float(alpha), float(beta), out, fmts[A.dtype], _stream_ptr(stream)))
    return C


def gemm_quant_i8_raw(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, in_type: int, Q: int, ldq: int,
                      alpha: float, bias: Optional[int], bias_dtype: int, activation: int, row_scale: Optional[int],
                      zero_point: int, stream: int, variant: int = 0) -> int:
    """Pointer-level call of the quantising entry point; returns the status."""
    return lib().gemm_quant_i8(M, N, K, A, lda, B, ldb, in_type, Q, ldq, alpha, bias, bias_dtype, activation,
                               row_scale, zero_point, stream, variant)


def gemm_quant_i8(A, B, Q, alpha: float = 1.0, *, row_scale, zero_point: int = 0, bias=None, activation="none",
                  M: Optional[int] = None, N: Optional[int] = None, K: Optional[int] = None, stream=None,
                  variant: int = 0):
    """Q = saturate_int8(rne(act(alpha*A*B + bias[j]) * row_scale[i] + zero_point)) on the GPU.
    A, B: bf16 or float8 (both the same) CUDA tensors in gemm_bf16's storage
    convention; Q: int8 (N, ldq); row_scale: contiguous fp32 CUDA tensor of
    at least M values."""
    import torch
    kinds = {torch.bfloat16: IN_BF16, torch.float8_e4m3fn: IN_E4M3, torch.float8_e5m2: IN_E5M2}
    if not (A.is_cuda and B.is_cuda and Q.is_cuda and row_scale.is_cuda):
        raise ValueError("A, B, Q and row_scale must be CUDA tensors")
    if A.dtype not in kinds or B.dtype != A.dtype:
        raise ValueError("A and B must both be bfloat16, float8_e4m3fn or float8_e5m2")
    if Q.dtype != torch.int8 or row_scale.dtype != torch.float32 or row_scale.dim() != 1:
        raise ValueError("Q must be int8 and row_scale 1-D float32")
    for t in (A, B, Q):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("A, B, Q must be 2-D with unit inner stride")
    M = Q.shape[1] if M is None else M
    N = Q.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    if Q.shape[0] < N or row_scale.shape[0] < M or (K > 0 and (A.shape[0] < M or B.shape[0] < N)):
        raise ValueError("tensor shapes smaller than M/N")
    if bias is None:
        bptr, bkind = None, BIAS_NONE
    else:
        if not bias.is_cuda or bias.dim() != 1 or bias.stride(0) != 1 or bias.shape[0] < N:
            raise ValueError("bias must be a contiguous 1-D CUDA tensor of at least N values")
        bkind = BIAS_F32 if bias.dtype == torch.float32 else BIAS_BF16 if bias.dtype == torch.bfloat16 else None
        if bkind is None:
            raise ValueError("bias must be float32 or bfloat16")
        bptr = bias.data_ptr()
    act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
    st = gemm_quant_i8_raw(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), kinds[A.dtype], Q.data_ptr(),
                           Q.stride(0), float(alpha), bptr, bkind, act, row_scale.data_ptr(), int(zero_point),
                           _stream_ptr(stream), variant)
    _check(st)
    return Q


def gemm_bf16_layout_raw(M: int, N: int, K: int, A: int, lda: int, a_layout: int, B: int, ldb: int, b_layout: int,
                         C: int, ldc: int, alpha: float, beta: float, out_dtype: int, stream: int,
                         variant: int = 0) -> int:
    """Pointer-level call of the any-layout entry point; returns the status."""
    return lib().gemm_bf16_layout(M, N, K, A, lda, a_layout, B, ldb, b_layout, C, ldc, alpha, beta, out_dtype,
                                  stream, variant)


def gemm_bf16_layout(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, a_col: bool = False, b_row: bool = False,
                     M: Optional[int] = None, N: Optional[int] = None, K: Optional[int] = None, stream=None,
                     variant: int = 0):
    """C = alpha * A * B + beta * C with A row-major (M, lda) or, with a_col,
    column-major (K, lda); B column-major (N, ldb) or, with b_row, row-major
    (K, ldb).  C as in gemm_bf16."""
    import torch
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("A, B and C must be CUDA tensors")
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise ValueError("A and B must be bfloat16")
    if C.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("C must be float32 or bfloat16")
    for t in (A, B, C):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("A, B, C must be 2-D with unit inner stride")
    M = C.shape[1] if M is None else M
    N = C.shape[0] if N is None else N
    K = (A.shape[0] if a_col else A.shape[1]) if K is None else K
    out = OUT_F32 if C.dtype == torch.float32 else OUT_BF16
    st = gemm_bf16_layout_raw(M, N, K, A.data_ptr(), A.stride(0), COL_MAJOR if a_col else ROW_MAJOR, B.data_ptr(),
                              B.stride(0), ROW_MAJOR if b_row else COL_MAJOR, C.data_ptr(), C.stride(0), float(alpha),
                              float(beta), out, _stream_ptr(stream), variant)
    _check(st)
    return C


def autotune(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, a_col: bool = False, b_row: bool = False,
             M: Optional[int] = None, N: Optional[int] = None, K: Optional[int] = None, iters: int = 10,
             flush=None, stream=None) -> tuple[int, float]:
    """Time every variant built for this problem on these tensors (storage
    convention of gemm_bf16 / gemm_bf16_layout / gemm_fp8) and remember the
    fastest for later automatic calls.  Returns (variant, microseconds).
    ``flush``: an optional CUDA tensor larger than L2, written before every
    timed call (cold-call timing).  C is overwritten."""
    import torch
    kinds = {torch.bfloat16: IN_BF16, torch.float8_e4m3fn: IN_E4M3, torch.float8_e5m2: IN_E5M2}
    if A.dtype not in kinds or B.dtype != A.dtype:
        raise ValueError("A and B must both be bfloat16, float8_e4m3fn or float8_e5m2")
    if C.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("C must be float32 or bfloat16")
    M = C.shape[1] if M is None else M
    N = C.shape[0] if N is None else N
    K = (A.shape[0] if a_col else A.shape[1]) if K is None else K
    best = ctypes.c_int(0)
    us = ctypes.c_float(0.0)
    st = lib().tcgemm_autotune(M, N, K, A.data_ptr(), A.stride(0), COL_MAJOR if a_col else ROW_MAJOR, B.data_ptr(),
                               B.stride(0), ROW_MAJOR if b_row else COL_MAJOR, kinds[A.dtype], C.data_ptr(),
                               C.stride(0), float(alpha), float(beta),
                               OUT_F32 if C.dtype == torch.float32 else OUT_BF16, int(iters),
                               None if flush is None else flush.data_ptr(),
                               0 if flush is None else flush.numel() * flush.element_size(), _stream_ptr(stream),
                               ctypes.byref(best), ctypes.byref(us))
    _check(st)
    return best.value, us.value


def autotune_lookup(M: int, N: int, K: int, in_type: int = 0, out_dtype: int = 1, a_col: bool = False,
                    b_row: bool = False, beta_nonzero: bool = False) -> int:
    return lib().tcgemm_autotune_lookup(M, N, K, in_type, out_dtype, COL_MAJOR if a_col else ROW_MAJOR,
                                        ROW_MAJOR if b_row else COL_MAJOR, int(beta_nonzero))


def autotune_clear() -> None:
    lib().tcgemm_autotune_clear()


def autotune_set(M: int, N: int, K: int, variant: int, in_type: int = 0, out_dtype: int = 1, a_col: bool = False,
                 b_row: bool = False, beta_nonzero: bool = False) -> None:
    """Record `variant` as the tuned choice for this problem (0 removes it)."""
    _check(lib().tcgemm_autotune_set(M, N, K, in_type, out_dtype, COL_MAJOR if a_col else ROW_MAJOR,
                                     ROW_MAJOR if b_row else COL_MAJOR, int(beta_nonzero), variant))


def autotune_save(path: str) -> int:
    """Write the tuned-choice table to a text file; returns the number of choices."""
    n = int(lib().tcgemm_autotune_save(str(path).encode()))
    if n < 0:
        raise TcgemmError(1, last_error())
    return n


def autotune_load(path: str) -> int:
    """Add the choices stored by autotune_save; returns how many were read."""
    n = int(lib().tcgemm_autotune_load(str(path).encode()))
    if n < 0:
        raise TcgemmError(1, last_error())
    return n


def check_device_status(stream=None) -> tuple[int, int]:
    where = ctypes.c_uint32(0)
    st = lib().tcgemm_check_device_status(_stream_ptr(stream), ctypes.byref(where))
    return st, where.value


def selftest_withheld_load(A, B, C, *, M: int, N: int, K: int, variant: int, timeout_ns: int,
                           stream=None) -> int:
    """tcgemm_selftest_withheld_load on torch tensors laid out as gemm_bf16's
    (C fp32); returns the status code (5 = TCGEMM_ERR_TIMEOUT expected)."""
    return int(lib().tcgemm_selftest_withheld_load(M, N, K, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1],
                                                   C.data_ptr(), C.shape[1], variant, timeout_ns,
                                                   _stream_ptr(stream)))


def selftest_timeout(timeout_ns: int, stream=None) -> int:
    return lib().tcgemm_selftest_timeout(_stream_ptr(stream), int(timeout_ns))


def launch_count() -> int:
    return int(lib().tcgemm_launch_count())


def pick_variant(M: int, N: int, K: int, num_sms: int) -> int:
    return int(lib().tcgemm_pick_variant(M, N, K, num_sms))


PLAN_KEYS = ["grid", "cluster", "tiles_m", "tiles_n", "bm", "bn", "num_kb", "smem", "tiles_dp",
             "sk_tiles", "sk_iters", "ws_bytes", "group_m", "variant", "cta_group", "grid_m", "grid_n",
             "stream_k", "arows", "swap", "ks", "hilbert"]


def plan(M: int, N: int, K: int, variant: int = 0, num_sms: int = 152, in_kind: int = 0, a_col: bool = False,
         b_row: bool = False) -> dict:
    """Launch plan for a device with `num_sms` SMs (host only; assumes every
    pair / 4-cluster of SMs can be resident).  in_kind 1: 8-bit operands;
    a_col / b_row: the layouts of gemm_bf16_layout."""
    out = (ctypes.c_int64 * len(PLAN_KEYS))()
    if in_kind or a_col or b_row:
        _check(lib().tcgemm_plan_kind(M, N, K, variant, in_kind, COL_MAJOR if a_col else ROW_MAJOR,
                                      ROW_MAJOR if b_row else COL_MAJOR, num_sms, out))
    else:
        _check(lib().tcgemm_plan(M, N, K, variant, num_sms, out))
    return dict(zip(PLAN_KEYS, [int(v) for v in out]))


def plan_device(M: int, N: int, K: int, variant: int = 0) -> dict:
    """The plan gemm_bf16 uses on the current device."""
    out = (ctypes.c_int64 * len(PLAN_KEYS))()
    _check(lib().tcgemm_plan_device(M, N, K, variant, out))
    return dict(zip(PLAN_KEYS, [int(v) for v in out]))


def device_info() -> dict:
    out = (ctypes.c_int64 * 4)()
    _check(lib().tcgemm_device_info(out))
    return {"sms": int(out[0]), "max_pairs": int(out[1]), "device": int(out[3])}


def gemm_bf16_noalloc_raw(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                          alpha: float, beta: float, out_dtype: int, stream: int, variant: int = 0) -> int:
    """Pointer-level call of the allocation-free entry point (fixed scratch
    array inside the library); returns the status."""
    return lib().gemm_bf16_noalloc(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant)


def noalloc_scratch_bytes() -> int:
    return int(lib().tcgemm_noalloc_scratch_bytes())


def noalloc_fits(M: int, N: int, K: int, variant: int = 0, num_sms: int = 152) -> bool:
    """Whether gemm_bf16_noalloc's fixed scratch holds this problem's plan
    on a device with num_sms SMs (host only)."""
    r = int(lib().tcgemm_noalloc_fits(M, N, K, variant, num_sms))
    if r < 0:
        raise TcgemmError(1, "bad arguments")
    return r == 1


def workspace_bytes(M: int, N: int, K: int, variant: int = 0, num_sms: int = 152) -> int:
    return int(lib().tcgemm_workspace_bytes(M, N, K, variant, num_sms))


def gemm_bf16_ws_raw(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                     alpha: float, beta: float, out_dtype: int, stream: int, variant: int,
                     workspace: int, workspace_bytes: int) -> int:
    """Pointer-level call with a caller-owned workspace; returns the status."""
    return lib().gemm_bf16_ws(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, stream, variant,
                              workspace, workspace_bytes)


UNIT_KEYS = ["tile", "kb0", "kb1", "slot", "sk_tile", "piece", "npieces"]


def units(M: int, N: int, K: int, variant: int, num_sms: int, cluster: int) -> list:
    """The work units of one cluster under the host plan (the kernel's own
    iterator, run on the host)."""
    n = int(lib().tcgemm_units(M, N, K, variant, num_sms, cluster, 0, (ctypes.c_int32 * 1)()))
    if n < 0:
        raise ValueError("bad arguments")
    buf = (ctypes.c_int32 * max(1, 7 * n))()
    lib().tcgemm_units(M, N, K, variant, num_sms, cluster, n, buf)
    return [dict(zip(UNIT_KEYS, buf[7 * i:7 * i + 7])) for i in range(n)]


def tile_order(tiles_m: int, tiles_n: int, group_m: int, count: Optional[int] = None):
    count = tiles_m * tiles_n if count is None else count
    tm = (ctypes.c_int32 * count)()
    tn = (ctypes.c_int32 * count)()
    _check(lib().tcgemm_tile_order(tiles_m, tiles_n, group_m, count, tm, tn))
    return list(tm), list(tn)


def tile_order_hilbert(tiles_m: int, tiles_n: int, count: Optional[int] = None):
    """The Hilbert visiting order (tcgemm_tile_order_hilbert): tile rows and columns."""
    count = tiles_m * tiles_n if count is None else count
    tm = (ctypes.c_int32 * max(count, 1))()
    tn = (ctypes.c_int32 * max(count, 1))()
    _check(lib().tcgemm_tile_order_hilbert(tiles_m, tiles_n, count, tm, tn))
    return list(tm)[:count], list(tn)[:count]


def version() -> int:
    return int(lib().tcgemm_version())
