"""CPU oracle for C = alpha*A*B + beta*C (bf16 in, fp64 sum, one rounding out).

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline / reference leg may import this module.  The CUDA
library never imports, links or calls it, and it shares no code with the CUDA
library: the arithmetic lives in ``gemm_oracle.c`` (plain C, compiled with gcc)
and this file only marshals numpy arrays into it.

Every function cites the passage it follows in ``gemm_oracle.c``'s header:
the product and layouts from the H100 work log "在 H100 上超越 cuBLAS：一份工作日志"
(sections "Simon 博客的快速回顾" and "实验设置"), and the alpha/beta update
from the "DeepGEMM" article, section 1.1; the fused bias + activation
epilogue from the same article, section 6.1; FP8 inputs (section 6.3) in the
OCP E4M3 / E5M2 formats; the per-token int8 quantisation of section 6.2 (the
readings taken where the article is silent are listed in ``gemm_oracle.c``'s
header).

Parity pins for this oracle live in ``tests/test_oracle_pins.py``.  The fp32
accumulation order of the GPU is a hardware choice; it is covered only by the
tolerance, not by a pin ("parity unpinned" beyond the tolerance).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()

# Activation codes of gemm_oracle.c (its own numbering; callers use the names).
ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2, "gelu_tanh": 3}
# Input kinds of gemm_oracle.c: bf16 (uint16 bit arrays) or an FP8 format (uint8 arrays).
# in_format is one format name for both operands, or a pair (format of A,
# format of B).
FP8_KINDS = {"e4m3": 1, "e5m2": 2, ("e4m3", "e4m3"): 1, ("e5m2", "e5m2"): 2, ("e4m3", "e5m2"): 3,
             ("e5m2", "e4m3"): 4}


def lib_path(mutant: int = 0, build_dir: Optional[str] = None) -> str:
    d = build_dir or _BUILD
    name = "liboracle.so" if mutant == 0 else f"liboracle_mut{mutant}.so"
    return os.path.join(d, name)


def build(mutant: int = 0, build_dir: Optional[str] = None, force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math, so every double
    operation rounds as written).  Returns the path of the shared object."""
    out = lib_path(mutant, build_dir)
    with _lock:
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            return out
        os.makedirs(os.path.dirname(out), exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off",
               f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class Oracle:
    """ctypes view of one compiled oracle (the real one or a planted mutant)."""

    def __init__(self, path: str):
        self.path = path
        L = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        L.oracle_gemm_f64.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, ctypes.c_int,
                                      ctypes.c_float, ctypes.c_float, p, ctypes.c_int]
        L.oracle_gemm_f64.restype = ctypes.c_int
        L.oracle_gemm_sampled_f64.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, ctypes.c_int,
                                              ctypes.c_float, ctypes.c_float, i64, p, p, p]
        L.oracle_gemm_sampled_f64.restype = ctypes.c_int
        L.oracle_gemm_epi_f64.argtypes = [i64, i64, i64, p, i64, p, i64, ctypes.c_int, p, i64, ctypes.c_int,
                                          ctypes.c_float, ctypes.c_float, p, ctypes.c_int, ctypes.c_int,
                                          p, ctypes.c_int]
        L.oracle_gemm_epi_f64.restype = ctypes.c_int
        L.oracle_gemm_epi_sampled_f64.argtypes = [i64, i64, i64, p, i64, p, i64, ctypes.c_int, p, i64,
                                                  ctypes.c_int, ctypes.c_float, ctypes.c_float, p, ctypes.c_int,
                                                  ctypes.c_int, i64, p, p, p]
        L.oracle_absdot_kind_sampled_f64.argtypes = [i64, i64, i64, p, i64, p, i64, ctypes.c_int, i64, p, p, p]
        L.oracle_absdot_kind_sampled_f64.restype = ctypes.c_int
        L.oracle_gemm_layout_f64.argtypes = [i64, i64, i64, p, i64, ctypes.c_int, p, i64, ctypes.c_int, p, i64,
                                             ctypes.c_int, ctypes.c_float, ctypes.c_float, p, ctypes.c_int]
        L.oracle_gemm_layout_f64.restype = ctypes.c_int
        L.oracle_gemm_layout_sampled_f64.argtypes = [i64, i64, i64, p, i64, ctypes.c_int, p, i64, ctypes.c_int, p,
                                                     i64, ctypes.c_int, ctypes.c_float, ctypes.c_float, i64, p, p, p,
                                                     ctypes.c_int]
        L.oracle_gemm_layout_sampled_f64.restype = ctypes.c_int
        L.oracle_quantize_i8.argtypes = [p, i64, i64, p, ctypes.c_int32, p]
        L.oracle_quantize_i8_sampled.argtypes = [p, i64, p, p, ctypes.c_int32, p]
        L.oracle_fp8_to_double.argtypes = [ctypes.c_uint8, ctypes.c_int]
        L.oracle_fp8_to_double.restype = ctypes.c_double
        L.oracle_gemm_epi_sampled_f64.restype = ctypes.c_int
        L.oracle_activation_array.argtypes = [p, p, i64, ctypes.c_int]
        L.oracle_absdot_sampled_f64.argtypes = [i64, i64, i64, p, i64, p, i64, i64, p, p, p]
        L.oracle_absdot_sampled_f64.restype = ctypes.c_int
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_round_bf16.restype = ctypes.c_uint16
        L.oracle_round_bf16_array.argtypes = [p, p, i64]
        L.oracle_round_f32_array.argtypes = [p, p, i64]
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_threads.argtypes = [ctypes.c_int]
        L.oracle_threads.restype = ctypes.c_int
        L.oracle_mutant_id.restype = ctypes.c_int
        self._L = L

    # -- helpers -------------------------------------------------------------
    @staticmethod
    def _ptr(a: Optional[np.ndarray]):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    @staticmethod
    def _cin(C_in, beta):
        # C_in is handed to the C code whenever the caller supplies it; the C
        # code itself decides (by the definition) not to read it when beta == 0.
        if C_in is None:
            return None, 0, 0
        C_in = np.ascontiguousarray(C_in)
        if C_in.dtype == np.uint16:
            return C_in, C_in.shape[1], 1
        if C_in.dtype == np.float32:
            return C_in, C_in.shape[1], 0
        raise TypeError("C_in must be float32 or bf16 bits (uint16)")

    @staticmethod
    def _bias(bias):
        """bias: None, float32 array (kind 1) or uint16 bf16 bits (kind 2), one
        value per column j of C."""
        if bias is None:
            return None, 0
        bias = np.ascontiguousarray(bias)
        if bias.dtype == np.float32:
            return bias, 1
        if bias.dtype == np.uint16:
            return bias, 2
        raise TypeError("bias must be float32 or bf16 bits (uint16)")

    @staticmethod
    def _operands(A, B, in_format):
        """A, B as contiguous arrays plus the C code's input kind: uint16 arrays
        hold bf16 bits; uint8 arrays hold FP8 codes of ``in_format``."""
        A = np.ascontiguousarray(A)
        B = np.ascontiguousarray(B)
        if A.dtype == np.uint8 and B.dtype == np.uint8:
            key = tuple(in_format) if isinstance(in_format, (list, tuple)) else in_format
            if key not in FP8_KINDS:
                raise ValueError("uint8 operands need in_format 'e4m3', 'e5m2' or a pair of them (A, B)")
            return A, B, FP8_KINDS[key]
        if in_format not in (None, "bf16"):
            raise ValueError("in_format given for bf16 operands")
        return np.ascontiguousarray(A, dtype=np.uint16), np.ascontiguousarray(B, dtype=np.uint16), 0

    @staticmethod
    def _act(act) -> int:
        return ACTIVATIONS[act] if isinstance(act, str) else int(act)

    @property
    def mutant(self) -> int:
        return self._L.oracle_mutant_id()

    def threads(self, n: int = 0) -> int:
        return self._L.oracle_threads(n)

    # -- the definition --------------------------------------------------------
    def gemm_f64(self, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray,
                 C_in: Optional[np.ndarray] = None, alpha: float = 1.0, beta: float = 0.0,
                 threads: int = 0, in_format: Optional[str] = None) -> np.ndarray:
        """D = alpha*A*B + beta*C_in in fp64.

        A: uint16 bf16 bits, shape (M, lda).  B: uint16, shape (N, ldb) (column
        j of B is row j).  C_in: (N, ldc) float32 or uint16 bf16 bits.
        Returns D as an (N, M) float64 array: D_arr[j, i] = D[i, j].  With
        uint8 operands (FP8 codes) ``in_format`` names their format.
        """
        A, B, kind = self._operands(A, B, in_format)
        assert A.shape[0] == M and B.shape[0] == N
        lda = A.shape[1] if A.ndim == 2 else K
        ldb = B.shape[1] if B.ndim == 2 else K
        cin, ldc, cin_bf16 = self._cin(C_in, beta)
        D = np.empty((N, M), dtype=np.float64)
        if kind == 0:
            rc = self._L.oracle_gemm_f64(M, N, K, self._ptr(A), lda, self._ptr(B), ldb,
                                         self._ptr(cin), max(ldc, M), cin_bf16,
                                         float(alpha), float(beta), self._ptr(D), int(threads))
        else:
            rc = self._L.oracle_gemm_epi_f64(M, N, K, self._ptr(A), lda, self._ptr(B), ldb, kind,
                                             self._ptr(cin), max(ldc, M), cin_bf16, float(alpha), float(beta),
                                             None, 0, 0, self._ptr(D), int(threads))
        if rc != 0:
            raise ValueError("oracle_gemm_f64: bad arguments")
        return D

    def gemm_epi_f64(self, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray,
                     C_in: Optional[np.ndarray] = None, alpha: float = 1.0, beta: float = 0.0,
                     bias: Optional[np.ndarray] = None, act="none", threads: int = 0,
                     in_format: Optional[str] = None) -> np.ndarray:
        """E = act(alpha*A*B + beta*C_in + bias[j]) in fp64, as an (N, M) array
        (the fused epilogue; see gemm_f64 for the layouts)."""
        A, B, kind = self._operands(A, B, in_format)
        assert A.shape[0] == M and B.shape[0] == N
        lda = A.shape[1] if A.ndim == 2 else K
        ldb = B.shape[1] if B.ndim == 2 else K
        cin, ldc, cin_bf16 = self._cin(C_in, beta)
        b, bkind = self._bias(bias)
        assert b is None or b.shape[0] >= N
        D = np.empty((N, M), dtype=np.float64)
        rc = self._L.oracle_gemm_epi_f64(M, N, K, self._ptr(A), lda, self._ptr(B), ldb, kind,
                                         self._ptr(cin), max(ldc, M), cin_bf16, float(alpha), float(beta),
                                         self._ptr(b), bkind, self._act(act), self._ptr(D), int(threads))
        if rc != 0:
            raise ValueError("oracle_gemm_epi_f64: bad arguments")
        return D

    def gemm_epi_sampled_f64(self, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray,
                             rows: np.ndarray, cols: np.ndarray,
                             C_in: Optional[np.ndarray] = None, alpha: float = 1.0, beta: float = 0.0,
                             bias: Optional[np.ndarray] = None, act="none",
                             in_format: Optional[str] = None) -> np.ndarray:
        A, B, kind = self._operands(A, B, in_format)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        cin, ldc, cin_bf16 = self._cin(C_in, beta)
        b, bkind = self._bias(bias)
        out = np.empty(rows.shape[0], dtype=np.float64)
        rc = self._L.oracle_gemm_epi_sampled_f64(M, N, K, self._ptr(A), A.shape[1], self._ptr(B), B.shape[1],
                                                 kind, self._ptr(cin), max(ldc, M), cin_bf16, float(alpha),
                                                 float(beta), self._ptr(b), bkind, self._act(act),
                                                 rows.shape[0], self._ptr(rows), self._ptr(cols),
                                                 self._ptr(out))
        if rc != 0:
            raise ValueError("oracle_gemm_epi_sampled_f64: bad arguments")
        return out

    def activation(self, x: np.ndarray, act) -> np.ndarray:
        """The oracle's activation function applied to fp64 values."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.float64)
        self._L.oracle_activation_array(self._ptr(x), self._ptr(out), x.size, self._act(act))
        return out

    def gemm_sampled_f64(self, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray,
                         rows: np.ndarray, cols: np.ndarray,
                         C_in: Optional[np.ndarray] = None, alpha: float = 1.0,
                         beta: float = 0.0, in_format: Optional[str] = None) -> np.ndarray:
        if in_format not in (None, "bf16"):
            return self.gemm_epi_sampled_f64(M, N, K, A, B, rows, cols, C_in, alpha, beta, in_format=in_format)
        A = np.ascontiguousarray(A, dtype=np.uint16)
        B = np.ascontiguousarray(B, dtype=np.uint16)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        cin, ldc, cin_bf16 = self._cin(C_in, beta)
        out = np.empty(rows.shape[0], dtype=np.float64)
        rc = self._L.oracle_gemm_sampled_f64(M, N, K, self._ptr(A), A.shape[1], self._ptr(B),
                                             B.shape[1], self._ptr(cin), max(ldc, M), cin_bf16,
                                             float(alpha), float(beta), rows.shape[0],
                                             self._ptr(rows), self._ptr(cols), self._ptr(out))
        if rc != 0:
            raise ValueError("oracle_gemm_sampled_f64: bad arguments")
        return out

    def absdot_sampled_f64(self, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray,
                           rows: np.ndarray, cols: np.ndarray, in_format: Optional[str] = None) -> np.ndarray:
        """G[i,j] = sum_k |A[i,k] * B[k,j]| at the given positions (fp64), the
        scale of the fp32-accumulation error bound."""
        A, B, kind = self._operands(A, B, in_format)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        out = np.empty(rows.shape[0], dtype=np.float64)
        rc = self._L.oracle_absdot_kind_sampled_f64(M, N, K, self._ptr(A), A.shape[1], self._ptr(B), B.shape[1],
                                                    kind, rows.shape[0], self._ptr(rows), self._ptr(cols),
                                                    self._ptr(out))
        if rc != 0:
            raise ValueError("oracle_absdot_sampled_f64: bad arguments")
        return out

    def round_bf16(self, d: np.ndarray) -> np.ndarray:
        d = np.ascontiguousarray(d, dtype=np.float64)
        out = np.empty(d.shape, dtype=np.uint16)
        self._L.oracle_round_bf16_array(self._ptr(d), self._ptr(out), d.size)
        return out

    def round_f32(self, d: np.ndarray) -> np.ndarray:
        d = np.ascontiguousarray(d, dtype=np.float64)
        out = np.empty(d.shape, dtype=np.float32)
        self._L.oracle_round_f32_array(self._ptr(d), self._ptr(out), d.size)
        return out

    def round_out(self, d: np.ndarray, out_dtype: int) -> np.ndarray:
        """out_dtype 0 -> float32 array, 1 -> uint16 bf16 bits."""
        return self.round_f32(d) if out_dtype == 0 else self.round_bf16(d)

    def gemm_layout_f64(self, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray, a_col: bool, b_row: bool,
                        C_in: Optional[np.ndarray] = None, alpha: float = 1.0, beta: float = 0.0,
                        threads: int = 0) -> np.ndarray:
        """D for bf16 operands in any layout: A is (M, lda) row-major or, with
        a_col, (K, lda) column-major; B is (N, ldb) column-major or, with
        b_row, (K, ldb) row-major.  Returns D as an (N, M) array."""
        A = np.ascontiguousarray(A, dtype=np.uint16)
        B = np.ascontiguousarray(B, dtype=np.uint16)
        cin, ldc, cin_bf16 = self._cin(C_in, beta)
        D = np.empty((N, M), dtype=np.float64)
        rc = self._L.oracle_gemm_layout_f64(M, N, K, self._ptr(A), A.shape[1], int(a_col), self._ptr(B), B.shape[1],
                                            int(b_row), self._ptr(cin), max(ldc, M), cin_bf16, float(alpha),
                                            float(beta), self._ptr(D), int(threads))
        if rc != 0:
            raise ValueError("oracle_gemm_layout_f64: bad arguments")
        return D

    def gemm_layout_sampled_f64(self, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray, a_col: bool,
                                b_row: bool, rows: np.ndarray, cols: np.ndarray, C_in: Optional[np.ndarray] = None,
                                alpha: float = 1.0, beta: float = 0.0, absolute: bool = False) -> np.ndarray:
        """D (or, with absolute, G = sum |a*b|) at the given positions."""
        A = np.ascontiguousarray(A, dtype=np.uint16)
        B = np.ascontiguousarray(B, dtype=np.uint16)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        cin, ldc, cin_bf16 = self._cin(C_in, beta)
        out = np.empty(rows.shape[0], dtype=np.float64)
        rc = self._L.oracle_gemm_layout_sampled_f64(M, N, K, self._ptr(A), A.shape[1], int(a_col), self._ptr(B),
                                                    B.shape[1], int(b_row), self._ptr(cin), max(ldc, M), cin_bf16,
                                                    float(alpha), float(beta), rows.shape[0], self._ptr(rows),
                                                    self._ptr(cols), self._ptr(out), int(absolute))
        if rc != 0:
            raise ValueError("oracle_gemm_layout_sampled_f64: bad arguments")
        return out

    def quantize_i8(self, E: np.ndarray, row_scale: np.ndarray, zero_point: int) -> np.ndarray:
        """int8 codes of the quantising epilogue from E, an (N, M) array of
        epilogue values (the layout gemm_f64 returns); row_scale: M fp32."""
        E = np.ascontiguousarray(E, dtype=np.float64)
        N, M = E.shape
        sc = np.ascontiguousarray(row_scale, dtype=np.float32)
        assert sc.shape[0] >= M
        Q = np.empty((N, M), dtype=np.int8)
        self._L.oracle_quantize_i8(self._ptr(E), M, N, self._ptr(sc), int(zero_point), self._ptr(Q))
        return Q

    def quantize_i8_sampled(self, values: np.ndarray, rows: np.ndarray, row_scale: np.ndarray,
                            zero_point: int) -> np.ndarray:
        values = np.ascontiguousarray(values, dtype=np.float64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        sc = np.ascontiguousarray(row_scale, dtype=np.float32)
        out = np.empty(values.shape[0], dtype=np.int8)
        self._L.oracle_quantize_i8_sampled(self._ptr(values), values.shape[0], self._ptr(rows), self._ptr(sc),
                                           int(zero_point), self._ptr(out))
        return out

    def bf16_to_double(self, bits: int) -> float:
        return self._L.oracle_bf16_to_double(bits)

    def fp8_to_double(self, code: int, in_format: str) -> float:
        """The value of one FP8 code ('e4m3' or 'e5m2')."""
        return self._L.oracle_fp8_to_double(code, FP8_KINDS[in_format] - 1)


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The real (unmutated) oracle, compiled on first use."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
