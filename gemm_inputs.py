"""Seeded synthetic inputs for the bf16 GEMM, shared by the oracle tests, the
CUDA parity tests and the benchmark.

This module only draws numbers and lays them out in memory; it contains none
of the GEMM arithmetic.  Both sides of every parity check receive the very
same bytes from here.

Distribution: the H100 work log "在 H100 上超越 cuBLAS：一份工作日志", section
"实验设置" (experimental setup), initialises every matrix from a normal
distribution with mean 0 and standard deviation 1 and multiplies bf16
matrices with A row-major and B, C column-major.  We draw fp32 N(0,1) from torch's CPU generator seeded
with ``torch.manual_seed``-style explicit generators, then round to bf16 with
round-to-nearest-even (``Tensor.to(torch.bfloat16)``).

Memory layout convention (every tensor here lives on the host):

* ``A``: row-major M x K with leading dimension ``lda`` -> torch tensor of
  shape ``(M, lda)``; element A[i, k] is ``A[i, k]``.
* ``B``: column-major K x N with leading dimension ``ldb`` -> shape
  ``(N, ldb)``; element B[k, j] is ``B[j, k]``.
* ``C``: column-major M x N with leading dimension ``ldc`` -> shape
  ``(N, ldc)``; element C[i, j] is ``C[j, i]``.

Padding columns beyond K (or M for C) are filled with a fixed sentinel so a
kernel that reads them would produce a visibly wrong answer.

FP8 inputs (E4M3 or E5M2, the OCP 8-bit formats) are drawn the same way and
rounded with torch's conversion to ``float8_e4m3fn`` / ``float8_e5m2``
(round to nearest even); their padding holds the code 0x7F, a NaN in both.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

# bf16 bit pattern 0x7FC0 = quiet NaN.  Padding is filled with it so that any
# read of a padding element poisons the result.
PAD_BF16_BITS = 0x7FC0

OUT_F32 = 0
OUT_BF16 = 1

FP8_DTYPES = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
PAD_FP8_BITS = 0x7F  # NaN in E4M3 and in E5M2


@dataclasses.dataclass
class GemmCase:
    """One GEMM problem: shapes, strides, scalars and host tensors."""

    name: str
    M: int
    N: int
    K: int
    lda: int
    ldb: int
    ldc: int
    alpha: float
    beta: float
    out_dtype: int  # OUT_F32 or OUT_BF16
    A: torch.Tensor  # (M, lda) bf16 or FP8, host
    B: torch.Tensor  # (N, ldb) bf16 or FP8, host
    C_in: Optional[torch.Tensor]  # (N, ldc) out dtype, host; None when beta == 0
    in_format: object = "bf16"  # "bf16", "e4m3" or "e5m2" (A and B), or a pair of FP8 formats (A's, B's)
    a_col: bool = False  # A stored column-major: A is (K, lda), A[i, k] = A[k, i]
    b_row: bool = False  # B stored row-major: B is (K, ldb), B[k, j] = B[k, j]

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def out_torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.out_dtype == OUT_F32 else torch.bfloat16


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(rows: int, cols: int, seed: int, ld: Optional[int] = None) -> torch.Tensor:
    """(rows, ld) bf16 tensor; the first ``cols`` columns are N(0,1) rounded to
    bf16, the padding columns hold the NaN sentinel."""
    ld = cols if ld is None else ld
    vals = torch.randn((rows, cols), generator=_gen(seed), dtype=torch.float32)
    out = torch.empty((rows, ld), dtype=torch.bfloat16)
    if ld > cols:
        out.view(torch.int16)[:, cols:] = PAD_BF16_BITS
    out[:, :cols] = vals.to(torch.bfloat16)
    return out


def normal_f32(rows: int, cols: int, seed: int, ld: Optional[int] = None) -> torch.Tensor:
    ld = cols if ld is None else ld
    vals = torch.randn((rows, cols), generator=_gen(seed), dtype=torch.float32)
    out = torch.full((rows, ld), float("nan"), dtype=torch.float32)
    out[:, :cols] = vals
    return out


def integer_bf16(rows: int, cols: int, seed: int, lo: int = -4, hi: int = 4,
                 ld: Optional[int] = None) -> torch.Tensor:
    """Small integers drawn uniformly from [lo, hi] (exact in bf16)."""
    ld = cols if ld is None else ld
    vals = torch.randint(lo, hi + 1, (rows, cols), generator=_gen(seed), dtype=torch.int32)
    out = torch.empty((rows, ld), dtype=torch.bfloat16)
    if ld > cols:
        out.view(torch.int16)[:, cols:] = PAD_BF16_BITS
    out[:, :cols] = vals.to(torch.bfloat16)
    return out


def integer_out(rows: int, cols: int, seed: int, out_dtype: int, lo: int = -8, hi: int = 8,
                ld: Optional[int] = None) -> torch.Tensor:
    ld = cols if ld is None else ld
    vals = torch.randint(lo, hi + 1, (rows, cols), generator=_gen(seed), dtype=torch.int32)
    dt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
    out = torch.full((rows, ld), float("nan"), dtype=dt)
    out[:, :cols] = vals.to(dt)
    return out


def _fp8(vals: torch.Tensor, rows: int, cols: int, fmt: str, ld: int) -> torch.Tensor:
    out = torch.empty((rows, ld), dtype=FP8_DTYPES[fmt])
    if ld > cols:
        out.view(torch.uint8)[:, cols:] = PAD_FP8_BITS
    out[:, :cols] = vals.to(FP8_DTYPES[fmt])
    return out


def normal_fp8(rows: int, cols: int, seed: int, fmt: str, ld: Optional[int] = None) -> torch.Tensor:
    """(rows, ld) FP8 tensor: N(0,1) rounded to the format, NaN padding."""
    ld = cols if ld is None else ld
    return _fp8(torch.randn((rows, cols), generator=_gen(seed), dtype=torch.float32), rows, cols, fmt, ld)


def integer_fp8(rows: int, cols: int, seed: int, fmt: str, lo: int = -4, hi: int = 4,
                ld: Optional[int] = None) -> torch.Tensor:
    """Small integers from [lo, hi], exact in both FP8 formats for |x| <= 4."""
    ld = cols if ld is None else ld
    vals = torch.randint(lo, hi + 1, (rows, cols), generator=_gen(seed), dtype=torch.int32)
    return _fp8(vals.to(torch.float32), rows, cols, fmt, ld)


def relayout(case: GemmCase, a_col: bool, b_row: bool, lda: Optional[int] = None,
             ldb: Optional[int] = None) -> GemmCase:
    """The same logical A and B stored in another layout (column-major A as
    (K, lda) with lda >= M; row-major B as (K, ldb) with ldb >= N); padding
    holds the NaN sentinel.  Only bf16 operands."""
    assert case.in_format == "bf16" and not case.a_col and not case.b_row
    M, N, K = case.M, case.N, case.K
    A, B = case.A[:, :K], case.B[:, :K]
    if a_col:
        lda = round_up(max(M, 1), 8) if lda is None else lda
        At = torch.empty((K, lda), dtype=torch.bfloat16)
        At.view(torch.int16)[:] = PAD_BF16_BITS
        At[:, :M] = A.t()
        A, la = At, lda
    else:
        A, la = case.A, case.lda
    if b_row:
        ldb = round_up(max(N, 1), 8) if ldb is None else ldb
        Bt = torch.empty((K, ldb), dtype=torch.bfloat16)
        Bt.view(torch.int16)[:] = PAD_BF16_BITS
        Bt[:, :N] = B.t()
        B, lb = Bt, ldb
    else:
        B, lb = case.B, case.ldb
    return dataclasses.replace(case, A=A, B=B, lda=la, ldb=lb, a_col=a_col, b_row=b_row)


def as_u8(t: torch.Tensor) -> np.ndarray:
    """FP8 torch tensor -> numpy uint8 view of the same bytes."""
    assert t.element_size() == 1
    return t.contiguous().view(torch.uint8).numpy()


def as_bits(t: torch.Tensor) -> np.ndarray:
    """Operand bytes for the oracle: uint16 bf16 bits or uint8 FP8 codes."""
    return as_u8(t) if t.element_size() == 1 else as_u16(t)


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def make_case(name: str, M: int, N: int, K: int, *, alpha: float = 1.0, beta: float = 0.0,
              out_dtype: int = OUT_BF16, seed: int = 0, kind: str = "normal",
              lda: Optional[int] = None, ldb: Optional[int] = None,
              ldc: Optional[int] = None, in_format: str = "bf16") -> GemmCase:
    """Build a case.  Leading dimensions default to the smallest value the
    16-byte stride rule allows (K rounded up to 8 bf16 or 16 FP8 elements for
    A/B, M rounded up to 16 bytes for C)."""
    per16 = 8 if in_format == "bf16" else 16
    lda = round_up(max(K, 1), per16) if lda is None else lda
    ldb = round_up(max(K, 1), per16) if ldb is None else ldb
    esz = 4 if out_dtype == OUT_F32 else 2
    ldc = round_up(max(M, 1), 16 // esz) if ldc is None else ldc
    if in_format != "bf16":
        fa, fb = (in_format, in_format) if isinstance(in_format, str) else tuple(in_format)
        if kind == "normal":
            A = normal_fp8(M, K, seed * 1000 + 1, fa, lda)
            B = normal_fp8(N, K, seed * 1000 + 2, fb, ldb)
        elif kind == "integer":
            A = integer_fp8(M, K, seed * 1000 + 1, fa, ld=lda)
            B = integer_fp8(N, K, seed * 1000 + 2, fb, ld=ldb)
        else:
            raise ValueError(kind)
    elif kind == "normal":
        A = normal_bf16(M, K, seed * 1000 + 1, lda)
        B = normal_bf16(N, K, seed * 1000 + 2, ldb)
    elif kind == "integer":
        A = integer_bf16(M, K, seed * 1000 + 1, ld=lda)
        B = integer_bf16(N, K, seed * 1000 + 2, ld=ldb)
    else:
        raise ValueError(kind)
    C_in = None
    if beta != 0.0:
        if kind == "integer":
            C_in = integer_out(N, M, seed * 1000 + 3, out_dtype, ld=ldc)
        elif out_dtype == OUT_F32:
            C_in = normal_f32(N, M, seed * 1000 + 3, ldc)
        else:
            C_in = normal_bf16(N, M, seed * 1000 + 3, ldc)
    return GemmCase(name, M, N, K, lda, ldb, ldc, float(alpha), float(beta), out_dtype,
                    A, B, C_in, in_format)


# The five workloads: square 256 (fp32 out), the square 4096 headline shape,
# square 8192 with a beta = 0.5 epilogue over an N(0,1) C, a shape that is no
# multiple of any tile, and a skinny weight-streaming shape.  Seeds are
# 1000 * index + {1, 2, 3} for A, B and C_in.
CONFIGS = {
    "s256": dict(M=256, N=256, K=256, alpha=1.0, beta=0.0, out_dtype=OUT_F32, seed=0),
    "s4k": dict(M=4096, N=4096, K=4096, alpha=1.0, beta=0.0, out_dtype=OUT_BF16, seed=1),
    "s8k": dict(M=8192, N=8192, K=8192, alpha=1.0, beta=0.5, out_dtype=OUT_BF16, seed=2),
    "edge": dict(M=4000, N=4100, K=4104, alpha=1.0, beta=0.0, out_dtype=OUT_F32, seed=3),
    "skinny": dict(M=64, N=8192, K=8192, alpha=1.0, beta=0.0, out_dtype=OUT_BF16, seed=4),
}


def config_case(name: str, kind: str = "normal") -> GemmCase:
    c = CONFIGS[name]
    return make_case(name, c["M"], c["N"], c["K"], alpha=c["alpha"], beta=c["beta"],
                     out_dtype=c["out_dtype"], seed=c["seed"], kind=kind)


def slab_bounds(n_total: int, world: int, rank: int, align: int = 1) -> tuple[int, int]:
    """Columns [n0, n1) of an n_total-column output that rank `rank` of
    `world` owns: contiguous slabs in rank order, each a multiple of `align`
    columns except possibly the last, as even as that allows (a rank may get
    none when n_total is small)."""
    if world < 1 or not 0 <= rank < world or align < 1 or n_total < 0:
        raise ValueError("bad slab arguments")
    units = (n_total + align - 1) // align
    u0 = units * rank // world
    u1 = units * (rank + 1) // world
    return min(n_total, u0 * align), min(n_total, u1 * align)


def slab_seed(seed: int, rank: int) -> int:
    """Seed of rank `rank`'s slab of a matrix whose slab 0 uses `seed` (so a
    one-rank job draws exactly the single-GPU workload)."""
    return int(seed) if rank == 0 else int(seed) + 7919 * rank


def column_slab_case(name: str, world: int, rank: int) -> GemmCase:
    """Rank `rank`'s part of one GEMM that is `world` times wider than the
    named workload: C = alpha*A*B + beta*C with M x (N*world) output, A
    replicated on every rank, and this rank holding the contiguous columns
    [rank*N, (rank+1)*N) of B and C (drawn from their own seeds; rank 0's
    slab is the named workload itself)."""
    c = CONFIGS[name]
    case = config_case(name)
    if rank == 0:
        return case
    s = c["seed"]
    M, N, K = c["M"], c["N"], c["K"]
    B = normal_bf16(N, K, slab_seed(s * 1000 + 2, rank), case.ldb)
    C_in = None
    if case.beta != 0.0:
        C_in = (normal_f32(N, M, slab_seed(s * 1000 + 3, rank), case.ldc) if case.out_dtype == OUT_F32
                else normal_bf16(N, M, slab_seed(s * 1000 + 3, rank), case.ldc))
    return dataclasses.replace(case, B=B, C_in=C_in)


def as_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 view of the same bytes."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_indices(M: int, N: int, count: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """Deterministic (row, col) sample that always includes the four corners,
    the last row and column, and random interior points."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, size=count))
    cols = list(rng.integers(0, N, size=count))
    extra = [(0, 0), (M - 1, 0), (0, N - 1), (M - 1, N - 1)]
    for j in rng.integers(0, N, size=16):
        extra.append((M - 1, int(j)))
    for i in rng.integers(0, M, size=16):
        extra.append((int(i), N - 1))
    for (i, j) in extra:
        rows.append(i)
        cols.append(j)
    return np.asarray(rows, dtype=np.int64), np.asarray(cols, dtype=np.int64)


def cell_sample_indices(M: int, N: int, cell_m: int, cell_n: int, per_cell: int,
                        seed: int) -> tuple[np.ndarray, np.ndarray]:
    """``per_cell`` random (row, col) positions inside every cell of a
    cell_m x cell_n grid laid over the M x N output, plus the corners, so that
    every tile of any tiling with tiles that are multiples of the cell is
    sampled."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for i0 in range(0, M, cell_m):
        hi = min(M, i0 + cell_m)
        for j0 in range(0, N, cell_n):
            hj = min(N, j0 + cell_n)
            rows.extend(rng.integers(i0, hi, size=per_cell).tolist())
            cols.extend(rng.integers(j0, hj, size=per_cell).tolist())
    for (i, j) in [(0, 0), (M - 1, 0), (0, N - 1), (M - 1, N - 1)]:
        rows.append(i)
        cols.append(j)
    return np.asarray(rows, dtype=np.int64), np.asarray(cols, dtype=np.int64)
