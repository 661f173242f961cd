"""GPU parity of the quantising epilogue (gemm_quant_i8: int8 codes of
act(alpha*A*B + bias) * row_scale[i] + zero_point, the "DeepGEMM" article's
section 6.2) against the oracle, through the C ABI.

The code is an integer decided by floating point.  The oracle decides it in
the kernel's precision (the value rounded to fp32, one fp32 fused multiply-add,
ties to even), but its value is the exact one while the GPU's carries the
fp32 accumulation error, so the two may land on different sides of a rounding
boundary.  What is unique is compared exactly: every code whose exact value
x*scale + zero_point lies farther from a boundary k + 1/2 than the GEMM error
bound (tests/parity.py, times |scale|) must match; the others may differ by
one.  Integer inputs with power-of-two scales are bit-exact.  Q is guarded
like C (bytes around it and the ldq padding rows must stay untouched).
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import parity

pytestmark = pytest.mark.gpu

VARIANTS = [int(v) for v in os.environ.get("QUANT_VARIANTS", "0,2,4,5,6,7").split(",")]
GUARD = 4096
SENT = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()


def _case(name, M, N, K, fmt, seed, kind="normal"):
    alpha = 1.0 if kind == "integer" else float(np.float32(1.0 / math.sqrt(max(K, 1))))
    ldq = gi.round_up(max(M, 1), 16) + (16 if M % 3 == 0 else 0)
    case = gi.make_case(name, M, N, K, alpha=alpha, beta=0.0, out_dtype=gi.OUT_F32, seed=seed, kind=kind,
                        in_format=fmt)
    return case, ldq


def run_quant(case, ldq, scale, zp, bias=None, act="none", variant=0):
    import tensor_core_matmul_gb300 as tc
    n = case.N * ldq
    buf = torch.full((n + 2 * GUARD,), SENT, dtype=torch.int8, device="cuda")
    Q = buf[GUARD:GUARD + n].view(case.N, ldq)
    before = buf.clone()
    tc.gemm_quant_i8(case.A.cuda(), case.B.cuda(), Q, case.alpha, row_scale=scale.cuda(), zero_point=zp,
                     bias=None if bias is None else bias.cuda(), activation=act, M=case.M, N=case.N, K=case.K,
                     variant=variant)
    torch.cuda.synchronize()
    st, where = tc.check_device_status()
    assert st == 0, f"device status {st} (role {where})"
    assert torch.equal(buf[:GUARD], before[:GUARD]) and torch.equal(buf[-GUARD:], before[-GUARD:]), "write outside Q"
    if ldq > case.M:
        assert torch.equal(Q[:, case.M:], before[GUARD:GUARD + n].view(case.N, ldq)[:, case.M:]), "write into padding"
    return Q[:, :case.M].cpu().numpy()


def compare_codes(o, case, got, scale, zp, bias=None, act="none", rows=None, cols=None, exact=False, what=""):
    fmt = None if case.in_format == "bf16" else case.in_format
    A, B = gi.as_bits(case.A), gi.as_bits(case.B)
    b = None if bias is None else (bias.numpy() if bias.dtype == torch.float32 else gi.as_u16(bias))
    if rows is None:
        cols, rows = np.divmod(np.arange(case.M * case.N, dtype=np.int64), case.M)
    E = o.gemm_epi_sampled_f64(case.M, case.N, case.K, A, B, rows, cols, None, case.alpha, 0.0, bias=b, act=act,
                               in_format=fmt)
    want = o.quantize_i8_sampled(E, rows, scale.numpy(), zp)
    g = got[cols, rows].astype(np.int32)
    w = want.astype(np.int32)
    if exact:
        bad = g != w
        assert not bad.any(), (what, np.argwhere(bad)[:5].ravel(), g[bad][:5], w[bad][:5])
        return
    s = scale.numpy().astype(np.float64)[rows]
    G = o.absdot_sampled_f64(case.M, case.N, case.K, A, B, rows, cols, in_format=fmt)
    S = o.gemm_sampled_f64(case.M, case.N, case.K, A, B, rows, cols, in_format=fmt)
    bb = 0.0 if b is None else np.abs(parity.bf16_to_f64(b[cols]) if b.dtype == np.uint16 else b[cols].astype(np.float64))
    L = parity.LIPSCHITZ[act]
    e_x = L * (abs(case.alpha) * case.K * parity.ACC_UNIT * G + 2.0 ** -22 * (abs(case.alpha) * np.abs(S) + bb)) \
        + parity.ACT_FN_REL * np.abs(E)
    v = E * s + zp
    margin = np.abs(s) * e_x + 2.0 ** -22 * np.abs(v) + 1e-30
    dist = np.abs(v - np.floor(v) - 0.5)  # distance to the nearest k + 1/2
    inside = (v > -128.5 - margin) & (v < 127.5 + margin)
    unique = ~inside | (dist > margin)
    bad_unique = unique & (g != w)
    assert not bad_unique.any(), (what, int(bad_unique.sum()), g[bad_unique][:5], w[bad_unique][:5],
                                  v[bad_unique][:5])
    assert np.all(np.abs(g - w) <= 1), what


def make_scale(M, seed, pow2=False):
    g = torch.Generator().manual_seed(seed)
    if pow2:
        return torch.pow(2.0, torch.randint(-3, 3, (M,), generator=g).to(torch.float32))
    return (torch.rand(M, generator=g, dtype=torch.float32) * 60.0 + 4.0)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("fmt", ["bf16", "e4m3"])
@pytest.mark.parametrize("act", ["none", "gelu"])
def test_quant_small_shapes(oracle_lib, variant, fmt, act):
    """Ragged shapes, per-row scales that spread the values over the int8
    range (so saturation happens too), a zero point, bias."""
    for n, (M, N, K, zp) in enumerate([(200, 300, 320, 0), (129, 520, 200, -5), (48, 260, 640, 7)]):
        case, ldq = _case(f"q{n}", M, N, K, fmt, seed=900 + n)
        scale = make_scale(M, 950 + n)
        bias = torch.randn(N, generator=torch.Generator().manual_seed(960 + n))
        got = run_quant(case, ldq, scale, zp, bias, act, variant)
        compare_codes(oracle_lib, case, got, scale, zp, bias, act, what=f"v{variant} {fmt} {act} {case.name}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_quant_integer_exact(oracle_lib, variant, fmt):
    """Integer inputs and bias, power-of-two row scales: every value is exact
    and so is every code."""
    case, ldq = _case("q_int", 300, 270, 500, fmt, seed=910, kind="integer")
    scale = make_scale(case.M, 970, pow2=True)
    bias = torch.randint(-40, 41, (case.N,), generator=torch.Generator().manual_seed(971)).to(torch.float32)
    got = run_quant(case, ldq, scale, 3, bias, "relu", variant)
    compare_codes(oracle_lib, case, got, scale, 3, bias, "relu", exact=True, what=f"v{variant} {fmt} integer")


def test_quant_stream_k(oracle_lib):
    """Stream-K shapes: the codes come out of the reduction kernel."""
    import tensor_core_matmul_gb300 as tc
    for n, (M, N, K) in enumerate([(600, 700, 8192), (40, 1000, 8192)]):
        assert tc.binding.plan_device(M, N, K, 0)["stream_k"] == 1
        case, ldq = _case(f"q_sk{n}", M, N, K, "bf16", seed=920 + n)
        scale = make_scale(M, 980 + n)
        got = run_quant(case, ldq, scale, 1)
        compare_codes(oracle_lib, case, got, scale, 1, what=f"stream-K {case.name}")
        assert np.array_equal(got, run_quant(case, ldq, scale, 1))


def test_quant_k_zero(oracle_lib):
    case, ldq = _case("q_k0", 70, 90, 0, "bf16", seed=930)
    scale = make_scale(70, 990)
    bias = torch.randn(90, generator=torch.Generator().manual_seed(991))
    compare_codes(oracle_lib, case, run_quant(case, ldq, scale, 2, bias, "relu"), scale, 2, bias, "relu",
                  what="K=0")


@pytest.mark.parametrize("config,fmt", [("s4k", "e4m3"), ("skinny", "bf16"), ("edge", "bf16")])
def test_quant_full_size_sampled(oracle_lib, config, fmt):
    c = gi.CONFIGS[config]
    case, ldq = _case(config, c["M"], c["N"], c["K"], fmt, seed=c["seed"])
    scale = make_scale(case.M, 995)
    got = run_quant(case, ldq, scale, -3)
    rows, cols = gi.cell_sample_indices(case.M, case.N, 128, 128, 2, seed=13)
    compare_codes(oracle_lib, case, got, scale, -3, rows=rows, cols=cols, what=f"{config} {fmt}")
