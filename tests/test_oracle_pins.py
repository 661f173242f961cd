"""Pins for the CPU oracle: checks against facts fixed by the pages' definition
and by mathematics, not by the oracle itself.

The pages print no worked numerical example, so the pins are:
  * exact brute force with Python integers on integer-valued bf16 inputs,
  * numpy's float64 matmul (an independent library routine) on N(0,1) inputs,
  * identity and permutation matrices, all-ones and rank-1 closed forms,
  * the bf16 rounding table in tests/golden/bf16_encodings.txt, derived by
    hand from the bf16 format, plus torch's fp32 -> bf16 conversion where the
    value is exactly a float,
  * beta == 0 never reading C, K == 0, and the N(0, K) statistics of the
    product of N(0,1) matrices,
  * for the fused bias + activation epilogue: exact brute force with
    integer inputs and biases through ReLU, the activations against
    independent library routines (torch.relu, scipy's normal distribution
    function for GELU, torch's tanh-approximated GELU), and the identity
    act(x) - act(-x) = x that ReLU and both GELUs satisfy,
  * for FP8 inputs: the hand-derived code table in
    tests/golden/fp8_encodings.txt, every one of the 256 codes of each format
    against torch's float8 -> float32 conversion, exact integer brute force and
    numpy's float64 matmul on the decoded values,
  * for the int8 quantising epilogue: the hand-derived table in
    tests/golden/quant_i8.txt (ties, saturation, zero point before rounding,
    the fp32 decision) and exact integer brute force through the GEMM,
  * for the other operand layouts: the same logical matrices stored
    transposed give bit-identical D, and integer brute force in each layout.

Each pin is a plain function of an ``Oracle`` so that ``test_planted_mistakes``
can run the same pins against oracle builds with one deliberate error each
and show that every error is caught.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import gemm_inputs as gi
import oracle as oracle_mod
from tests import parity

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _u16(t):
    return gi.as_u16(t)


def _cin_np(case):
    if case.C_in is None:
        return None
    if case.C_in.dtype == torch.bfloat16:
        return _u16(case.C_in)
    return case.C_in.numpy()


def _as_int(bits: np.ndarray) -> np.ndarray:
    """Integer-valued bf16 bits -> Python-int object array, decoded by the
    format (no oracle code): value = (-1)^s * 1.f * 2^(e-127)."""
    out = np.empty(bits.shape, dtype=object)
    flat = bits.reshape(-1)
    res = out.reshape(-1)
    for n, b in enumerate(flat):
        b = int(b)
        s, e, f = b >> 15, (b >> 7) & 0xFF, b & 0x7F
        if e == 0 and f == 0:
            v = Fraction(0)
        else:
            v = Fraction(128 + f, 128) * (Fraction(2) ** (e - 127))
        res[n] = -v if s else v
    return out


def _run(o, case):
    return o.gemm_f64(case.M, case.N, case.K, _u16(case.A), _u16(case.B), _cin_np(case),
                      case.alpha, case.beta)


# ---------------------------------------------------------------- pins ------

def pin_integer_bruteforce(o):
    """Integer inputs: every product and partial sum is an exact integer, so
    the oracle's D must equal the exact rational alpha*sum + beta*C."""
    shapes = [(5, 7, 9, 1.0, 0.0), (3, 2, 17, 2.0, 0.5), (6, 4, 3, -1.5, 0.5),
              (1, 9, 12, 1.0, -2.0), (9, 1, 1, 0.25, 1.0)]
    for n, (M, N, K, alpha, beta) in enumerate(shapes):
        case = gi.make_case(f"int{n}", M, N, K, alpha=alpha, beta=beta, out_dtype=gi.OUT_F32,
                            seed=100 + n, kind="integer", lda=K + 3, ldb=K + 5, ldc=M + 2)
        D = _run(o, case)
        A = _as_int(_u16(case.A)[:, :K])
        B = _as_int(_u16(case.B)[:, :K])  # row j = column j of B
        Cin = None if case.C_in is None else case.C_in.numpy()
        for i in range(M):
            for j in range(N):
                s = sum((A[i, k] * B[j, k] for k in range(K)), Fraction(0))
                want = Fraction(alpha) * s
                if beta != 0.0:
                    want += Fraction(beta) * Fraction(float(Cin[j, i]))
                assert D[j, i] == float(want), (n, i, j, D[j, i], want)
        rows, cols = np.divmod(np.arange(M * N), N)
        G = o.absdot_sampled_f64(M, N, K, _u16(case.A), _u16(case.B), rows, cols)
        for s_, (i, j) in enumerate(zip(rows, cols)):
            want = sum((abs(A[i, k] * B[j, k]) for k in range(K)), Fraction(0))
            assert G[s_] == float(want), (n, i, j, G[s_], want)


def pin_numpy_f64(o):
    """N(0,1) inputs: numpy's float64 matmul computes the same sum in another
    order; the two agree within the fp64 summation error bound."""
    M, N, K = 37, 29, 300
    case = gi.make_case("np", M, N, K, alpha=1.25, beta=0.5, out_dtype=gi.OUT_F32, seed=7,
                        lda=K + 8, ldb=K + 16, ldc=M + 3)
    D = _run(o, case)
    A = case.A[:, :K].to(torch.float64).numpy()
    B = case.B[:, :K].to(torch.float64).numpy()
    C = case.C_in[:, :M].to(torch.float64).numpy()
    ref = 1.25 * (B @ A.T) + 0.5 * C            # (N, M) layout, like D
    bound = 2 * K * 2.0 ** -52 * (np.abs(B) @ np.abs(A).T) * 1.25 + 1e-300
    assert np.all(np.abs(D - ref) <= bound + 2.0 ** -52 * np.abs(ref)), np.max(np.abs(D - ref))


def pin_identity_and_permutation(o):
    """A = I gives D = B exactly; B = I gives A laid out column-major; a row
    permutation of I permutes the rows of B."""
    K = 24
    Bcase = gi.make_case("b", K, 11, K, seed=3, out_dtype=gi.OUT_F32, lda=K, ldb=K + 8)
    eye = torch.eye(K, dtype=torch.bfloat16)
    D = o.gemm_f64(K, 11, K, _u16(eye), _u16(Bcase.B))
    B64 = Bcase.B[:, :K].to(torch.float64).numpy()     # (N, K): B64[j, k] = B[k, j]
    assert np.array_equal(D, B64)                      # D[j, i] = B[i, j]
    Acase = gi.make_case("a", 13, K, K, seed=4, out_dtype=gi.OUT_F32, lda=K + 8, ldb=K)
    D = o.gemm_f64(13, K, K, _u16(Acase.A), _u16(eye))
    A64 = Acase.A[:, :K].to(torch.float64).numpy()     # (M, K)
    assert np.array_equal(D, A64.T)                    # D[j, i] = A[i, j]
    perm = np.random.default_rng(5).permutation(K)
    P = torch.zeros((K, K), dtype=torch.bfloat16)
    P[np.arange(K), perm] = 1.0                        # P[i, perm[i]] = 1
    D = o.gemm_f64(K, 11, K, _u16(P), _u16(Bcase.B))
    assert np.array_equal(D, B64[:, perm])             # D[i, j] = B[perm[i], j]


def pin_closed_forms(o):
    """All-ones: D = alpha*K + beta*C.  Rank one: A[i,k] = u_i w_k,
    B[k,j] = w_k v_j gives D = u_i v_j sum_k w_k^2 (all small powers of two,
    so exact)."""
    M, N, K = 7, 5, 33
    ones_a = torch.ones((M, K), dtype=torch.bfloat16)
    ones_b = torch.ones((N, K), dtype=torch.bfloat16)
    C = gi.integer_out(N, M, 9, gi.OUT_F32)
    D = o.gemm_f64(M, N, K, _u16(ones_a), _u16(ones_b), C.numpy(), 3.0, -0.5)
    assert np.array_equal(D, 3.0 * K - 0.5 * C.numpy().astype(np.float64))
    u = np.array([1, -2, 4, 0.5, -1, 8, 2], dtype=np.float64)
    v = np.array([2, 1, -0.25, 4, -1], dtype=np.float64)
    w = np.array([(-1) ** k * 2.0 ** (k % 5 - 2) for k in range(K)])
    A = torch.tensor(np.outer(u, w), dtype=torch.bfloat16)
    B = torch.tensor(np.outer(v, w), dtype=torch.bfloat16)  # row j = column j
    D = o.gemm_f64(M, N, K, _u16(A), _u16(B))
    assert np.array_equal(D, np.outer(v, u) * float(np.sum(w * w)))
    r, c = np.divmod(np.arange(M * N), N)
    G = o.absdot_sampled_f64(M, N, K, _u16(A), _u16(B), r, c)
    assert np.array_equal(G, np.abs(u[r] * v[c]) * float(np.sum(w * w)))


def pin_bf16_rounding(o):
    """One RNE rounding from double straight to bf16: hand-derived table,
    then torch's fp32 -> bf16 conversion on values that are exactly floats."""
    path = os.path.join(GOLDEN, "bf16_encodings.txt")
    for line in open(path):
        line = line.split("#")[0].split()
        if not line:
            continue
        x, want = float.fromhex(line[0]), int(line[1], 16)
        got = int(o.round_bf16(np.array([x]))[0])
        assert got == want, (line[0], hex(got), hex(want))
    vals = torch.randn(20000, generator=torch.Generator().manual_seed(11)) * 1000
    vals = torch.cat([vals, torch.randn(5000, generator=torch.Generator().manual_seed(12)) * 1e-38])
    want = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = o.round_bf16(vals.to(torch.float64).numpy())
    assert np.array_equal(got, want)
    f = o.round_f32(np.array([1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, 1e39]))
    assert f[0] == np.float32(1.0) and f[1] == np.float32(1.0 + 2.0 ** -22) and np.isinf(f[2])


def pin_beta_zero_ignores_c(o):
    """beta == 0: C_in is not read, so a C full of NaN leaves no trace."""
    case = gi.make_case("nan", 9, 6, 20, seed=13, out_dtype=gi.OUT_F32)
    C = np.full((6, 9), np.nan, dtype=np.float32)
    D = o.gemm_f64(9, 6, 20, _u16(case.A), _u16(case.B), C, 1.0, 0.0)
    assert np.all(np.isfinite(D))
    D0 = o.gemm_f64(9, 6, 20, _u16(case.A), _u16(case.B))
    assert np.array_equal(D, D0)


def pin_k_zero(o):
    """K == 0: the empty sum is 0, so D = beta * C_in."""
    C = gi.integer_out(4, 3, 17, gi.OUT_F32).numpy()
    A = np.zeros((3, 8), dtype=np.uint16)
    B = np.zeros((4, 8), dtype=np.uint16)
    D = o.gemm_f64(3, 4, 0, A, B, C, 1.0, 0.5)
    assert np.array_equal(D, 0.5 * C.astype(np.float64))
    assert np.array_equal(o.gemm_f64(3, 4, 0, A, B), np.zeros((4, 3)))


def pin_statistics(o):
    """A, B with i.i.d. N(0,1) entries: each entry of A*B has mean 0 and
    variance K, so the sample standard deviation is close to sqrt(K)."""
    case = gi.make_case("st", 192, 160, 256, seed=19, out_dtype=gi.OUT_F32)
    D = _run(o, case)
    assert abs(D.std() / np.sqrt(256) - 1.0) < 0.03, D.std()
    assert abs(D.mean()) < 0.1 * np.sqrt(256)


def pin_sampled_matches_full(o):
    """The per-entry routine and the full routine evaluate the same
    definition; at sampled positions they agree bit for bit, and the rounding
    routine agrees with the full output."""
    case = gi.make_case("smp", 33, 47, 70, alpha=0.75, beta=-1.0, seed=23, out_dtype=gi.OUT_BF16,
                        lda=72, ldb=80, ldc=40)
    D = _run(o, case)
    rows, cols = gi.sample_indices(33, 47, 50, 1)
    s = o.gemm_sampled_f64(33, 47, 70, _u16(case.A), _u16(case.B), rows, cols, _cin_np(case),
                           case.alpha, case.beta)
    assert np.array_equal(s, D[cols, rows])


def pin_epilogue_integer_bruteforce(o):
    """Integer inputs and an integer bias: D + bias[j] is an exact integer
    (or half-integer), so act none / relu must give exactly
    max(alpha*S + beta*C + bias[j], 0) computed with rationals.  Shapes are
    not square and the bias array is longer than N (its extra entries must
    never be read), so a bias indexed by row would show."""
    shapes = [(5, 3, 9, 2.0, 0.0, "f32"), (3, 6, 17, -1.0, 0.5, "bf16"), (7, 4, 5, 1.0, -2.0, "f32"),
              (2, 9, 12, 0.5, 1.0, "bf16")]
    rng = np.random.default_rng(5)
    for n, (M, N, K, alpha, beta, bkind) in enumerate(shapes):
        case = gi.make_case(f"eint{n}", M, N, K, alpha=alpha, beta=beta, out_dtype=gi.OUT_F32,
                            seed=300 + n, kind="integer", lda=K + 1, ldb=K + 2, ldc=M + 1)
        vals = rng.integers(-40, 41, size=M + N + 3).astype(np.float32)
        bias = vals if bkind == "f32" else _u16(torch.from_numpy(vals).to(torch.bfloat16))
        A = _as_int(_u16(case.A)[:, :K])
        B = _as_int(_u16(case.B)[:, :K])
        Cin = None if case.C_in is None else case.C_in.numpy()
        for act in ("none", "relu"):
            E = o.gemm_epi_f64(M, N, K, _u16(case.A), _u16(case.B), _cin_np(case), alpha, beta,
                               bias=bias, act=act)
            for i in range(M):
                for j in range(N):
                    s = sum((A[i, k] * B[j, k] for k in range(K)), Fraction(0))
                    want = Fraction(alpha) * s + Fraction(int(vals[j]))
                    if beta != 0.0:
                        want += Fraction(beta) * Fraction(float(Cin[j, i]))
                    if act == "relu":
                        want = max(want, Fraction(0))
                    assert E[j, i] == float(want), (n, act, i, j, E[j, i], want)
        rows, cols = gi.sample_indices(M, N, 12, 3)
        smp = o.gemm_epi_sampled_f64(M, N, K, _u16(case.A), _u16(case.B), rows, cols, _cin_np(case),
                                     alpha, beta, bias=bias, act="relu")
        assert np.array_equal(smp, E[cols, rows])


def _act_grid():
    x = np.concatenate([np.linspace(-9.0, 9.0, 3601), [0.0, -0.0, 1e-30, -1e-30, 1e-8, -1e-8, 30.0, -30.0]])
    return x


def pin_activations_library(o):
    """The activations against independent library routines in float64:
    torch.relu; x * Phi(x) with Phi from scipy.special.ndtr (the normal
    distribution function, computed there without cancellation); torch's
    GELU with approximate='tanh' where its own 1 + tanh form does not cancel
    (x >= -3), and within its absolute rounding error below that."""
    from scipy.special import ndtr
    x = _act_grid()
    xt = torch.from_numpy(x)
    relu = o.activation(x, "relu")
    assert np.array_equal(relu, torch.relu(xt).numpy())
    gelu = o.activation(x, "gelu")
    ref = x * ndtr(x)
    assert np.allclose(gelu, ref, rtol=1e-12, atol=0.0), np.max(np.abs(gelu - ref) / np.maximum(np.abs(ref), 1e-300))
    gt = o.activation(x, "gelu_tanh")
    reft = torch.nn.functional.gelu(xt, approximate="tanh").numpy()
    hi = x >= -3.0
    assert np.allclose(gt[hi], reft[hi], rtol=1e-12, atol=1e-15)
    assert np.all(np.abs(gt[~hi] - reft[~hi]) <= 1e-14 * np.abs(x[~hi]))
    # The approximation stays close to the exact GELU (a published property
    # of the tanh form: the two differ by well under 1e-3 everywhere).
    assert np.max(np.abs(gt - ref)) < 1e-3


def pin_activation_odd_identity(o):
    """act(x) - act(-x) = x for ReLU (exactly) and for both GELUs (x*Phi(x)
    + x*Phi(-x) = x; the tanh form's (1 + tanh z)/2 + (1 - tanh z)/2 = 1), to
    within fp64 rounding.  Also act(0) = 0 and act(x) -> x for large x."""
    x = _act_grid()
    x = x[np.isfinite(x)]
    for act in ("relu", "gelu", "gelu_tanh"):
        d = o.activation(x, act) - o.activation(-x, act)
        tol = 0.0 if act == "relu" else 4e-16 * np.abs(x) + 1e-300
        assert np.all(np.abs(d - x) <= tol), act
        assert o.activation(np.array([0.0]), act)[0] == 0.0
        assert abs(o.activation(np.array([30.0]), act)[0] - 30.0) < 1e-12


def _fp8_values(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Decode FP8 codes with torch's conversion (a library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(gi.FP8_DTYPES[fmt])
    return t.to(torch.float32).numpy().astype(np.float64)


def pin_fp8_codes(o):
    """The FP8 decoder against the hand-derived table and, for all 256 codes
    of each format, against torch's float8 conversion."""
    for line in open(os.path.join(GOLDEN, "fp8_encodings.txt")):
        line = line.split("#")[0].split()
        if not line:
            continue
        fmt, code, val = line[0], int(line[1], 16), line[2]
        got = o.fp8_to_double(code, fmt)
        if val == "nan":
            assert np.isnan(got), (fmt, hex(code), got)
        else:
            want = float(val)
            assert got == want and np.signbit(got) == np.signbit(want), (fmt, hex(code), got, want)
    codes = np.arange(256, dtype=np.uint8)
    for fmt in ("e4m3", "e5m2"):
        got = np.array([o.fp8_to_double(int(c), fmt) for c in codes])
        want = _fp8_values(codes, fmt)
        same = (got == want) | (np.isnan(got) & np.isnan(want))
        assert same.all(), (fmt, codes[~same][:5], got[~same][:5], want[~same][:5])


def pin_fp8_integer_bruteforce(o):
    """Integer-valued FP8 inputs (exact in both formats): D must equal the
    exact rational alpha*sum + beta*C, with padded leading dimensions."""
    for n, (M, N, K, alpha, beta, fmt) in enumerate([(5, 7, 9, 1.0, 0.0, "e4m3"), (4, 3, 33, -2.0, 0.5, "e5m2"),
                                                      (3, 6, 17, 0.5, 1.0, "e4m3")]):
        case = gi.make_case(f"f8int{n}", M, N, K, alpha=alpha, beta=beta, out_dtype=gi.OUT_F32, seed=700 + n,
                            kind="integer", lda=K + 16 - K % 16 + 16, ldb=K + 16 - K % 16, ldc=M + 3,
                            in_format=fmt)
        A8, B8 = gi.as_u8(case.A), gi.as_u8(case.B)
        D = o.gemm_f64(M, N, K, A8, B8, _cin_np(case), alpha, beta, in_format=fmt)
        A = _fp8_values(A8[:, :K], fmt)
        B = _fp8_values(B8[:, :K], fmt)
        Cin = None if case.C_in is None else case.C_in.numpy()
        for i in range(M):
            for j in range(N):
                s = sum((Fraction(int(A[i, k])) * Fraction(int(B[j, k])) for k in range(K)), Fraction(0))
                want = Fraction(alpha) * s
                if beta != 0.0:
                    want += Fraction(beta) * Fraction(float(Cin[j, i]))
                assert D[j, i] == float(want), (n, i, j, D[j, i], want)
        rows, cols = gi.sample_indices(M, N, 10, 5)
        smp = o.gemm_sampled_f64(M, N, K, A8, B8, rows, cols, _cin_np(case), alpha, beta, in_format=fmt)
        assert np.array_equal(smp, D[cols, rows])


def pin_fp8_numpy_f64(o):
    """N(0,1) FP8 inputs: numpy's float64 matmul of the torch-decoded values
    agrees within the fp64 summation bound."""
    for fmt in ("e4m3", "e5m2"):
        M, N, K = 23, 31, 200
        case = gi.make_case("f8np", M, N, K, alpha=0.75, beta=0.0, out_dtype=gi.OUT_F32, seed=710, in_format=fmt)
        A8, B8 = gi.as_u8(case.A), gi.as_u8(case.B)
        D = o.gemm_f64(M, N, K, A8, B8, None, 0.75, 0.0, in_format=fmt)
        A = _fp8_values(A8[:, :K], fmt)
        B = _fp8_values(B8[:, :K], fmt)
        ref = 0.75 * (B @ A.T)
        G = np.abs(B) @ np.abs(A).T
        assert np.all(np.abs(D - ref) <= K * 2.0 ** -52 * G + 1e-300), fmt
        absd = o.absdot_sampled_f64(M, N, K, A8, B8, np.array([0, M - 1]), np.array([N - 1, 0]), in_format=fmt)
        assert np.allclose(absd, [G[N - 1, 0], G[0, M - 1]], rtol=1e-12)


def pin_quant_table(o):
    rows = []
    for line in open(os.path.join(GOLDEN, "quant_i8.txt")):
        f = line.split("#")[0].split()
        if f:
            rows.append((float(f[0]), float(f[1]), int(f[2]), int(f[3])))
    for x, sc, zp, want in rows:
        got = int(o.quantize_i8(np.array([[x]]), np.array([sc], dtype=np.float32), zp)[0, 0])
        assert got == want, (x, sc, zp, got, want)


def _rne(q: Fraction) -> int:
    f = q.numerator // q.denominator
    r = q - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def pin_quant_gemm_integer(o):
    """Integer inputs, power-of-two row scales and an integer bias: every
    value is exact, so the codes must be the exact rationals rounded half to
    even and saturated (brute force with Python integers)."""
    M, N, K = 6, 5, 11
    case = gi.make_case("qint", M, N, K, alpha=1.0, beta=0.0, out_dtype=gi.OUT_F32, seed=900, kind="integer")
    scale = np.array([0.5, 0.25, 2.0, 1.0, 0.125, 4.0], dtype=np.float32)
    bias = np.arange(N + 2, dtype=np.float32) - 3
    for zp, act in ((0, "none"), (3, "relu"), (-7, "none")):
        E = o.gemm_epi_f64(M, N, K, _u16(case.A), _u16(case.B), None, 1.0, 0.0, bias=bias, act=act)
        Q = o.quantize_i8(E, scale, zp)
        A = _as_int(_u16(case.A)[:, :K])
        B = _as_int(_u16(case.B)[:, :K])
        for i in range(M):
            for j in range(N):
                e = sum((A[i, k] * B[j, k] for k in range(K)), Fraction(0)) + Fraction(int(bias[j]))
                if act == "relu":
                    e = max(e, Fraction(0))
                want = max(-128, min(127, _rne(e * Fraction(float(scale[i])) + zp)))
                assert int(Q[j, i]) == want, (zp, act, i, j, int(Q[j, i]), want)
        rows, cols = gi.sample_indices(M, N, 8, 1)
        smp = o.quantize_i8_sampled(E[cols, rows], rows, scale, zp)
        assert np.array_equal(smp, Q[cols, rows])


def pin_layouts(o):
    """The four operand layouts: the same logical matrices stored the other
    way give the identical D (same terms, same order), and an integer case in
    each layout equals exact brute force over the logical matrices."""
    case = gi.make_case("lay", 13, 9, 21, alpha=1.5, beta=0.5, out_dtype=gi.OUT_F32, seed=950)
    D0 = o.gemm_f64(case.M, case.N, case.K, _u16(case.A), _u16(case.B), _cin_np(case), case.alpha, case.beta)
    icase = gi.make_case("layi", 7, 5, 10, alpha=2.0, beta=0.0, out_dtype=gi.OUT_F32, seed=951, kind="integer")
    A = _as_int(_u16(icase.A)[:, :icase.K])
    B = _as_int(_u16(icase.B)[:, :icase.K])
    for a_col in (False, True):
        for b_row in (False, True):
            r = gi.relayout(case, a_col, b_row, lda=case.M + 3 if a_col else None, ldb=case.N + 7 if b_row else None)
            D = o.gemm_layout_f64(case.M, case.N, case.K, _u16(r.A), _u16(r.B), a_col, b_row, _cin_np(case),
                                  case.alpha, case.beta)
            assert np.array_equal(D, D0), (a_col, b_row)
            rows, cols = gi.sample_indices(case.M, case.N, 10, 2)
            smp = o.gemm_layout_sampled_f64(case.M, case.N, case.K, _u16(r.A), _u16(r.B), a_col, b_row, rows, cols,
                                            _cin_np(case), case.alpha, case.beta)
            assert np.array_equal(smp, D0[cols, rows])
            ri = gi.relayout(icase, a_col, b_row)
            Di = o.gemm_layout_f64(icase.M, icase.N, icase.K, _u16(ri.A), _u16(ri.B), a_col, b_row, None, 2.0, 0.0)
            for i in range(icase.M):
                for j in range(icase.N):
                    want = 2 * sum((A[i, k] * B[j, k] for k in range(icase.K)), Fraction(0))
                    assert Di[j, i] == float(want), (a_col, b_row, i, j)


def pin_fp8_mixed_formats(o):
    """A in one FP8 format and B in the other: each operand is decoded in its
    own format.  Every FP8 value is exactly a bf16 value, so D must equal, bit
    for bit, the bf16 definition run on the torch-decoded values; and
    integer inputs give the exact rational result."""
    for n, (fa, fb) in enumerate((("e4m3", "e5m2"), ("e5m2", "e4m3"))):
        M, N, K = 9, 11, 70
        case = gi.make_case(f"f8mix{n}", M, N, K, alpha=1.25, beta=0.0, out_dtype=gi.OUT_F32, seed=720 + n,
                            in_format=(fa, fb))
        A8, B8 = gi.as_u8(case.A), gi.as_u8(case.B)
        D = o.gemm_f64(M, N, K, A8, B8, None, 1.25, 0.0, in_format=(fa, fb))
        A16 = gi.as_u16(torch.from_numpy(_fp8_values(A8[:, :K], fa).astype(np.float32)).to(torch.bfloat16))
        B16 = gi.as_u16(torch.from_numpy(_fp8_values(B8[:, :K], fb).astype(np.float32)).to(torch.bfloat16))
        assert np.array_equal(D, o.gemm_f64(M, N, K, A16, B16, None, 1.25, 0.0)), (fa, fb)
        icase = gi.make_case(f"f8mixi{n}", 4, 5, 33, alpha=1.0, beta=0.0, out_dtype=gi.OUT_F32, seed=730 + n,
                             kind="integer", in_format=(fa, fb))
        Ai, Bi = gi.as_u8(icase.A), gi.as_u8(icase.B)
        Di = o.gemm_f64(4, 5, 33, Ai, Bi, None, 1.0, 0.0, in_format=(fa, fb))
        Av, Bv = _fp8_values(Ai[:, :33], fa), _fp8_values(Bi[:, :33], fb)
        for i in range(4):
            for j in range(5):
                assert Di[j, i] == float(sum(Fraction(int(Av[i, k])) * Fraction(int(Bv[j, k])) for k in range(33)))


PINS = [pin_integer_bruteforce, pin_numpy_f64, pin_identity_and_permutation, pin_closed_forms,
        pin_bf16_rounding, pin_beta_zero_ignores_c, pin_k_zero, pin_statistics,
        pin_sampled_matches_full, pin_epilogue_integer_bruteforce, pin_activations_library,
        pin_activation_odd_identity, pin_fp8_codes, pin_fp8_integer_bruteforce, pin_fp8_numpy_f64,
        pin_quant_table, pin_quant_gemm_integer, pin_layouts, pin_fp8_mixed_formats]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(oracle_lib, pin):
    pin(oracle_lib)


MUTANTS = {
    1: "A read as column-major",
    2: "B read as row-major",
    3: "beta term dropped",
    4: "alpha and beta swapped",
    5: "last k term dropped",
    6: "beta term subtracted",
    7: "bf16 rounding truncates",
    8: "C_in read as row-major",
    9: "C_in read when beta == 0",
    10: "fp32 accumulation",
    11: "bias indexed by row",
    12: "activation applied before the bias",
    13: "GELU without the 1/sqrt(2) scaling",
    14: "tanh GELU without its cubic term",
    15: "bias added before alpha",
    16: "E4M3 subnormals scaled by 2^-10",
    17: "E5M2 decoded with E4M3's exponent bias",
    18: "quantisation truncates instead of rounding",
    19: "quantisation wraps instead of saturating",
    20: "zero point added after rounding",
    21: "column-major A read as row-major",
    22: "mixed FP8 formats: B decoded in A's format",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[m] for m in sorted(MUTANTS)])
def test_planted_mistakes_are_caught(tmp_path_factory, mutant):
    """Each oracle build with one planted error fails at least one pin."""
    d = str(tmp_path_factory.mktemp("mutants"))
    o = oracle_mod.Oracle(oracle_mod.build(mutant=mutant, build_dir=d))
    assert o.mutant == mutant
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake '{MUTANTS[mutant]}' passed every pin"


def test_ulp_distance_rules():
    """The bf16 comparison maps both zeros to 0 and counts ulps across 0."""
    d = parity.bf16_ulp_distance(np.array([0x0000, 0x3F80, 0x0001, 0x7F7F], dtype=np.uint16),
                                 np.array([0x8000, 0x3F81, 0x8001, 0x7F80], dtype=np.uint16))
    assert d.tolist() == [0, 1, 2, 1]
    with pytest.raises(AssertionError):
        parity.check_bf16(np.array([0x3F80], np.uint16), np.array([0x3F82], np.uint16))
    with pytest.raises(AssertionError):
        parity.check_f32(np.array([1.0 + 0.05]), np.array([1.0]), K=1)
    parity.check_f32(np.array([1.0 + 0.0009]), np.array([1.0]), K=1)
