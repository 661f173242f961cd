"""CPU checks of the cap on the bf16 second clause (parity.second_clause_cap)
on an N(0,1) problem, with emulated accumulators: each block of 16 products
is summed exactly (as one MMA step) and added to an fp32 accumulator.

* rounding to nearest, or truncating (the tensor cores' accumulation lies
  between the two): under the cap;
* an accumulator that keeps 2 fewer mantissa bits (an order- or
  precision-dependent mistake that costs a few ulps near zero): over the cap,
  although every one of its elements is within the worst-case bound of the
  second clause;
* 6 fewer bits: rejected by the comparison itself.  No GPU."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import gpu_harness as H
from tests import parity


def _accumulate(case: gi.GemmCase, mode: str, drop_bits: int = 0) -> np.ndarray:
    A = case.A.float().numpy()[:, :case.K].astype(np.float64)
    B = case.B.float().numpy()[:, :case.K].astype(np.float64)
    acc = np.zeros((case.N, case.M), dtype=np.float32)
    keep = np.uint32((0xFFFFFFFF << drop_bits) & 0xFFFFFFFF)
    for k0 in range(0, case.K, 16):
        s = acc.astype(np.float64) + B[:, k0:k0 + 16] @ A[:, k0:k0 + 16].T   # exact in float64
        r = s.astype(np.float32)                                               # round to nearest
        if mode == "truncate":
            over = np.abs(r.astype(np.float64)) > np.abs(s)
            r = np.where(over, np.nextafter(r, np.float32(0.0)), r).astype(np.float32)
        acc = (r.view(np.uint32) & keep).view(np.float32)
    return gi.as_u16(torch.from_numpy(acc).to(torch.bfloat16))


@pytest.fixture(scope="module")
def case():
    return gi.make_case("cap", 192, 256, 4096, alpha=1.0, beta=0.0, out_dtype=gi.OUT_BF16, seed=31)


def _cap(case) -> float:
    return parity.second_clause_cap(case.K) * case.M * case.N + 2


@pytest.mark.parametrize("mode", ["nearest", "truncate"])
def test_fp32_accumulation_is_under_the_cap(oracle_lib, case, mode):
    stats = H.compare_full(oracle_lib, case, _accumulate(case, mode), what=f"fp32 {mode}")
    assert stats["second_clause"] <= _cap(case), stats


def test_two_lost_bits_exceed_the_cap(oracle_lib, case):
    stats = H.compare_full(oracle_lib, case, _accumulate(case, "nearest", drop_bits=2), what="2 bits lost")
    assert stats["second_clause"] > _cap(case), stats


def test_six_lost_bits_fail_the_comparison(oracle_lib, case):
    with pytest.raises(AssertionError):
        H.compare_full(oracle_lib, case, _accumulate(case, "nearest", drop_bits=6), what="6 bits lost")
