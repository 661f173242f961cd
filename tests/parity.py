"""Comparison rules shared by the parity tests.

* fp32 output: |C - C_ref| <= 1e-3 * sqrt(K) * max(1, |C_ref|), elementwise.
* bf16 output: the two bit patterns, mapped to an ordered integer line, are at
  most 1 apart (within one bf16 ulp of the oracle's single rounding).
  Where the exact value is so small (cancellation) that the fp32 accumulator's
  own rounding error exceeds half a bf16 ulp, no fp32-accumulating kernel can
  meet that bar; there an element is also accepted if
      |C - D| <= ulp_bf16(D) + K * 2^-24 * G,   G = sum_k |A[i,k] B[k,j]|,
  the classical worst-case bound for a K-term floating-point sum in any
  order, plus the output rounding.  At most 0.5% (+2) of the elements may
  need this second clause, so a real bug cannot hide behind it.
* Integer-valued inputs: bit-exact.
* Fused epilogue E = act(D + bias): the activations are Lipschitz with
  constant L (1 for ReLU and none; 1.129 for both GELUs, the largest slope of
  x*Phi(x) and of its tanh form), so an error e in the value before the
  activation becomes at most L*e after it.  fp32 output:
      |C - E| <= L * 1e-3 * sqrt(K) * max(1, |D + bias|)  (+ 2^-20 |E| for the
      fp32 activation function's own error);
  bf16 output: within 1 ulp, or (second clause, same 0.5% (+2) cap)
      |C - E| <= ulp_bf16(E) + L * (|alpha| K 2^-24 G + 2^-22 (|alpha S| +
      |beta C| + |bias|)) + 2^-20 |E|,
  the accumulation bound plus the fp32 epilogue's few roundings.

C_ref is the oracle's fp64 value D (for fp32 output) or its bf16 rounding.

The check functions return a dict of statistics, so that a test can bound
how often the second clause was needed: ``size``, ``beyond_1ulp`` (bf16
elements more than one ulp from the oracle's rounding), ``second_clause``
(those accepted by the second clause), ``max_ulp`` (largest ordered-integer
distance) and, for fp32 output, ``max_err_over_tol``.
"""
from __future__ import annotations

import numpy as np


def bf16_ordered(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that increase with the value.
    +0 and -0 both map to 0; negative values map below zero."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(bf16_ordered(a_bits) - bf16_ordered(b_bits))


def f32_tolerance(ref: np.ndarray, K: int) -> np.ndarray:
    return 1e-3 * np.sqrt(max(K, 1)) * np.maximum(1.0, np.abs(ref))


def check_f32(got: np.ndarray, ref_f64: np.ndarray, K: int, what: str = "") -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref_f64, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return {"size": 0, "max_err_over_tol": 0.0}
    err = np.abs(got - ref)
    tol = f32_tolerance(ref, K)
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} fp32 outputs out of "
                             f"tolerance; first {idx.tolist()} got {got[bad][:5]} ref {ref[bad][:5]}")
    return {"size": int(got.size), "max_err_over_tol": float(np.max(err / tol))}


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (2^-133 below the normal range)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 7)


ACC_UNIT = 2.0 ** -24  # unit roundoff of the fp32 accumulator


def check_bf16(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = "", max_ulp: int = 1,
               fallback=None) -> dict:
    """``fallback(flat_indices) -> (D, G, K)`` supplies the exact value D and
    G = sum|a*b| at the elements that miss the 1-ulp bar (see module doc)."""
    got_bits = np.asarray(got_bits, dtype=np.uint16)
    ref_bits = np.asarray(ref_bits, dtype=np.uint16)
    assert got_bits.shape == ref_bits.shape
    if got_bits.size == 0:
        return {"size": 0, "beyond_1ulp": 0, "second_clause": 0, "max_ulp": 0}
    d = bf16_ulp_distance(got_bits, ref_bits)
    bad = d > max_ulp
    nan_got = (got_bits & 0x7FFF) > 0x7F80
    bad |= nan_got
    beyond = int(bad.sum())
    second = 0
    if bad.any() and fallback is not None and not nan_got.any():
        flat = np.flatnonzero(bad)
        limit = int(0.005 * got_bits.size) + 2
        if flat.size <= limit:
            D, G, K = fallback(flat)
            got = bf16_to_f64(got_bits.reshape(-1)[flat])
            ok = np.abs(got - D) <= bf16_ulp(D) + K * ACC_UNIT * G
            bad.reshape(-1)[flat[ok]] = False
            second = int(ok.sum())
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {got_bits.size} bf16 outputs more than "
                             f"{max_ulp} ulp away; first {idx.tolist()} got "
                             f"{[hex(x) for x in got_bits[bad][:5]]} ref {[hex(x) for x in ref_bits[bad][:5]]}")
    return {"size": int(got_bits.size), "beyond_1ulp": beyond, "second_clause": second, "max_ulp": int(d.max())}


def second_clause_cap(K: int) -> float:
    """Largest share of an N(0,1) workload's bf16 elements allowed to need
    the derived second clause (more than one ulp from the oracle's rounding,
    within the fp32 accumulation bound).

    Model: the fp32 accumulator (K/16 MMA additions into partial sums of size
    about sqrt(K)) carries an error e of standard deviation sigma ~ 2^-24 K/4.
    The bf16 result lands more than one ulp from the correct rounding only
    where |e| exceeds an ulp of D, i.e. |D| < 256 |e|; with D ~ N(0, K) that
    share is about (512 / sqrt(2 pi)) E|e| / sqrt(K) = 163 sigma / sqrt(K)
    = 2.4e-6 sqrt(K).  The cap is three times that (4.7e-4 at K = 4096,
    6.6e-4 at 8192): on the GB300 the full-size workloads need the clause for
    1.5e-4 (4096^3) and 3.4e-4 (8192^3) of their elements; emulated on the
    CPU (tests/test_second_clause_cap.py), an fp32 accumulator that rounds to
    nearest needs it for 2e-5, one that truncates for 2.4e-4, and one that
    keeps two fewer mantissa bits for 1e-3, over the cap although each of its
    elements is within the clause's worst-case bound."""
    sigma = 2.0 ** -24 * K / 4.0
    return 3.0 * 163.0 * sigma / np.sqrt(K)


LIPSCHITZ = {"none": 1.0, "relu": 1.0, "gelu": 1.13, "gelu_tanh": 1.13}
ACT_FN_REL = 2.0 ** -20  # allowance for the fp32 activation function's error (erfcf, expf: a few ulp)


def check_f32_epilogue(got: np.ndarray, E: np.ndarray, pre: np.ndarray, K: int, act: str, what: str = "") -> None:
    """fp32 output of the fused epilogue: E the oracle's act(D + bias), pre
    its D + bias (the value the activation is applied to)."""
    got = np.asarray(got, dtype=np.float64)
    E = np.asarray(E, dtype=np.float64)
    pre = np.asarray(pre, dtype=np.float64)
    assert got.shape == E.shape == pre.shape
    if got.size == 0:
        return
    tol = LIPSCHITZ[act] * f32_tolerance(pre, K) + ACT_FN_REL * np.abs(E)
    err = np.abs(got - E)
    bad = ~(err <= tol)
    bad &= ~(np.isnan(got) & np.isnan(E))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} fp32 outputs out of tolerance; "
                             f"first {idx.tolist()} got {got[bad][:5]} ref {E[bad][:5]}")


def check_bf16_bound(got_bits: np.ndarray, ref_bits: np.ndarray, bound_fn, what: str = "",
                     max_ulp: int = 1) -> dict:
    """As check_bf16, the second clause given as ``bound_fn(flat) -> (E,
    bound)``: an element is also accepted if |C - E| <= ulp_bf16(E) + bound."""
    got_bits = np.asarray(got_bits, dtype=np.uint16)
    ref_bits = np.asarray(ref_bits, dtype=np.uint16)
    assert got_bits.shape == ref_bits.shape
    if got_bits.size == 0:
        return {"size": 0, "beyond_1ulp": 0, "second_clause": 0, "max_ulp": 0}
    d = bf16_ulp_distance(got_bits, ref_bits)
    bad = d > max_ulp
    nan_got = (got_bits & 0x7FFF) > 0x7F80
    nan_ref = (ref_bits & 0x7FFF) > 0x7F80
    bad |= nan_got != nan_ref
    bad &= ~(nan_got & nan_ref)
    beyond = int(bad.sum())
    second = 0
    if bad.any():
        flat = np.flatnonzero(bad)
        if flat.size <= int(0.005 * got_bits.size) + 2:
            E, bound = bound_fn(flat)
            got = bf16_to_f64(got_bits.reshape(-1)[flat])
            ok = np.abs(got - E) <= bf16_ulp(E) + bound
            bad.reshape(-1)[flat[ok]] = False
            second = int(ok.sum())
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {got_bits.size} bf16 outputs more than "
                             f"{max_ulp} ulp away; first {idx.tolist()} got "
                             f"{[hex(x) for x in got_bits[bad][:5]]} ref {[hex(x) for x in ref_bits[bad][:5]]}")
    fin = ~(nan_got | nan_ref)
    return {"size": int(got_bits.size), "beyond_1ulp": beyond, "second_clause": second,
            "max_ulp": int(d[fin].max()) if fin.any() else 0}


def check_exact(got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    got = np.asarray(got)
    ref = np.asarray(ref)
    if got.dtype == np.uint16 or ref.dtype == np.uint16:
        eq = got.astype(np.uint16) == ref.astype(np.uint16)
    else:
        eq = got.astype(np.float64) == ref.astype(np.float64)
    if not eq.all():
        idx = np.argwhere(~eq)[:5]
        raise AssertionError(f"{what}: {int((~eq).sum())} of {got.size} outputs not bit-exact; "
                             f"first {idx.tolist()} got {got[~eq][:5]} ref {ref[~eq][:5]}")
