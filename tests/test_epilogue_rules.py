"""CPU checks of the fused-epilogue comparison rules (tests/parity.py): an
fp32 emulation of what the GPU epilogue computes passes them, and a result
with a planted mistake (the bias added along rows) fails them.  No GPU."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import test_gpu_epilogue as T


def _act32(x: np.ndarray, act: str) -> np.ndarray:
    from scipy.special import erfc
    x = x.astype(np.float32)
    if act == "relu":
        return np.where((x > 0) | np.isnan(x), x, np.float32(0.0))
    if act == "gelu":
        return (np.float32(0.5) * x * erfc(np.float32(-0.70710678) * x).astype(np.float32)).astype(np.float32)
    if act == "gelu_tanh":
        z = np.float32(0.7978845608) * (x + np.float32(0.044715) * x * x * x)
        return (x / (np.float32(1.0) + np.exp(np.float32(-2.0) * z))).astype(np.float32)
    return x


def _emulate(case: gi.GemmCase, bias_rows: np.ndarray, act: str):
    """fp32 product, fp32 epilogue, one rounding to the output type; the
    bias broadcast given by ``bias_rows`` (shape (N, 1) for the right axis)."""
    A = case.A.float().numpy()[:, :case.K]
    B = case.B.float().numpy()[:, :case.K]
    S = (B @ A.T).astype(np.float32)  # (N, M)
    v = np.float32(case.alpha) * S
    if case.beta != 0.0:
        v = v + np.float32(case.beta) * case.C_in.float().numpy()[:, :case.M]
    r = _act32((v + bias_rows).astype(np.float32), act)
    if case.out_dtype == gi.OUT_F32:
        return r
    return gi.as_u16(torch.from_numpy(r).to(torch.bfloat16))


@pytest.mark.parametrize("act", T.ACTS)
@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16], ids=["f32", "bf16"])
def test_rules_accept_fp32_epilogue_and_reject_row_bias(oracle_lib, act, out):
    case = T._case("rules", 129, 200, 320, out, 0.5, seed=3)
    bias = T.make_bias(case.N, "bf16", seed=1)
    b = bias.float().numpy()
    T.compare_epi(oracle_lib, case, _emulate(case, b[:, None], act), bias, act, what="fp32 emulation")
    with pytest.raises(AssertionError):
        T.compare_epi(oracle_lib, case, _emulate(case, b[None, :case.M], act), bias, act, what="row bias")
