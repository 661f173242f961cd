"""GPU parity of the fused epilogue, C = act(alpha*A*B + beta*C + bias[j])
(the "DeepGEMM" article, section 6.1: bias, then ReLU/GELU, inside the GEMM's
epilogue), through the C ABI entry point gemm_bf16_bias_act, against the
oracle's gemm_epi_f64 (fp64, one rounding).  Rules in tests/parity.py.

alpha = 1/sqrt(K) in the N(0,1) cases keeps the values near the activations'
curved region (|x| of order 1) instead of deep in their linear tails.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import gpu_harness as H
from tests import parity

pytestmark = pytest.mark.gpu

VARIANTS = [int(v) for v in os.environ.get("VARIANTS", "1,2,4,5,6,7").split(",")]
ACTS = ["relu", "gelu", "gelu_tanh", "none"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()


def make_bias(N: int, kind: str, seed: int, integer: bool = False) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    if integer:
        b = torch.randint(-40, 41, (N,), generator=g).to(torch.float32)
    else:
        b = torch.randn(N, generator=g, dtype=torch.float32)
    return b if kind == "f32" else b.to(torch.bfloat16)


def bias_np(b: torch.Tensor) -> np.ndarray:
    return b.numpy() if b.dtype == torch.float32 else gi.as_u16(b)


def run_epi(case: gi.GemmCase, bias, act: str, variant: int = 0) -> np.ndarray:
    import tensor_core_matmul_gb300 as tc
    g = H.GuardedC(case)
    tc.gemm_bf16_bias_act(case.A.cuda(), case.B.cuda(), g.C, case.alpha, case.beta,
                          bias=None if bias is None else bias.cuda(), activation=act,
                          M=case.M, N=case.N, K=case.K, variant=variant)
    torch.cuda.synchronize()
    st, where = tc.check_device_status()
    assert st == 0, f"device status {st} (role {where})"
    g.check_guards()
    return g.result_np()


def compare_epi(o, case: gi.GemmCase, got: np.ndarray, bias, act: str, rows=None, cols=None,
                exact: bool = False, what: str = ""):
    """got: (N, M) result.  rows/cols: positions to compare (all when None)."""
    A, B, cin = gi.as_u16(case.A), gi.as_u16(case.B), H.cin_np(case)
    b = None if bias is None else bias_np(bias)
    if rows is None:
        cols, rows = np.divmod(np.arange(case.M * case.N, dtype=np.int64), case.M)
    E = o.gemm_epi_sampled_f64(case.M, case.N, case.K, A, B, rows, cols, cin, case.alpha, case.beta,
                               bias=b, act=act)
    pre = o.gemm_epi_sampled_f64(case.M, case.N, case.K, A, B, rows, cols, cin, case.alpha, case.beta,
                                 bias=b, act="none")
    g = got[cols, rows]
    if case.out_dtype == gi.OUT_F32:
        if exact:
            parity.check_exact(g, o.round_f32(E), what)
        else:
            parity.check_f32_epilogue(g, E, pre, case.K, act, what)
        return
    ref = o.round_bf16(E)
    if exact:
        parity.check_exact(g, ref, what)
        return

    def bound(flat):
        r, c = rows[flat], cols[flat]
        G = o.absdot_sampled_f64(case.M, case.N, case.K, A, B, r, c)
        S = o.gemm_sampled_f64(case.M, case.N, case.K, A, B, r, c)
        bc = 0.0
        if case.beta != 0.0:
            bc = np.abs(case.beta * o.gemm_sampled_f64(case.M, case.N, 0, A, B, r, c, cin, 0.0, 1.0))
        bb = 0.0 if b is None else np.abs(parity.bf16_to_f64(b[c]) if b.dtype == np.uint16 else b[c].astype(np.float64))
        L = parity.LIPSCHITZ[act]
        e = L * (abs(case.alpha) * case.K * parity.ACC_UNIT * G
                 + 2.0 ** -22 * (abs(case.alpha) * np.abs(S) + bc + bb)) + parity.ACT_FN_REL * np.abs(E[flat])
        return E[flat], e
    parity.check_bf16_bound(g, ref, bound, what)


def _case(name, M, N, K, out, beta, seed, kind="normal", ldc=None):
    alpha = 1.0 if kind == "integer" else float(np.float32(1.0 / math.sqrt(max(K, 1))))
    return gi.make_case(name, M, N, K, alpha=alpha, beta=beta, out_dtype=out, seed=seed, kind=kind, ldc=ldc)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16], ids=["f32", "bf16"])
def test_epilogue_small_shapes(oracle_lib, variant, act, out):
    """Ragged shapes spanning several tiles in both directions, every variant,
    both bias types, beta on and off."""
    shapes = [(200, 300, 320, 0.0, "f32"), (129, 520, 200, 0.5, "bf16"), (48, 260, 640, 0.0, "bf16")]
    for n, (M, N, K, beta, bkind) in enumerate(shapes):
        case = _case(f"epi{n}", M, N, K, out, beta, seed=400 + 10 * n + out)
        bias = make_bias(N, bkind, seed=500 + n)
        got = run_epi(case, bias, act, variant)
        compare_epi(oracle_lib, case, got, bias, act, what=f"v{variant} {act} {case.name}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16], ids=["f32", "bf16"])
def test_epilogue_integer_exact(oracle_lib, variant, out):
    """Integer inputs and integer bias through ReLU: every intermediate is
    exact, so the result is bit-exact."""
    case = _case("epi_int", 300, 270, 500, out, 0.5, seed=410 + out, kind="integer")
    bias = make_bias(case.N, "bf16" if out else "f32", seed=510, integer=True)
    got = run_epi(case, bias, "relu", variant)
    compare_epi(oracle_lib, case, got, bias, "relu", exact=True, what=f"v{variant} int relu")


@pytest.mark.parametrize("act", ["gelu", "relu"])
def test_epilogue_stream_k(oracle_lib, act):
    """Shapes whose plan shares out k-blocks (stream-K): the epilogue runs in
    the reduction kernel, plain and transposed."""
    import tensor_core_matmul_gb300 as tc
    for n, (M, N, K, beta) in enumerate([(600, 700, 8192, 0.5), (40, 1000, 8192, 0.0)]):
        p = tc.binding.plan_device(M, N, K, 0)
        assert p["stream_k"] == 1, p
        case = _case(f"epi_sk{n}", M, N, K, gi.OUT_BF16, beta, seed=420 + n)
        bias = make_bias(N, "f32", seed=520 + n)
        got = run_epi(case, bias, act)
        compare_epi(oracle_lib, case, got, bias, act, what=f"stream-K {act} {case.name}")
        again = run_epi(case, bias, act)
        assert np.array_equal(got, again), "stream-K epilogue not repeatable"


def test_epilogue_k_zero(oracle_lib):
    """K == 0: act(beta*C + bias[j])."""
    for beta in (0.0, 0.75):
        case = _case("epi_k0", 70, 90, 0, gi.OUT_F32, beta, seed=430)
        bias = make_bias(case.N, "f32", seed=530)
        got = run_epi(case, bias, "gelu")
        compare_epi(oracle_lib, case, got, bias, "gelu", what=f"K=0 beta={beta}")


def test_epilogue_none_equals_plain_gemm():
    """No bias and no activation: the same bits as gemm_bf16."""
    case = _case("epi_plain", 333, 444, 555, gi.OUT_BF16, 0.5, seed=440)
    got = run_epi(case, None, "none")
    ref = H.run_case(case, 0).result_np()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("config,act", [("s4k", "gelu_tanh"), ("skinny", "gelu"), ("edge", "relu")])
def test_epilogue_full_size_sampled(oracle_lib, config, act):
    """Full-size workloads in the benchmark's launch configuration with the
    fused epilogue, checked at 2 positions in every 128 x 128 cell of C (so in
    every tile of every variant)."""
    c = gi.CONFIGS[config]
    case = gi.make_case(config, c["M"], c["N"], c["K"], alpha=float(np.float32(1.0 / math.sqrt(c["K"]))),
                        beta=c["beta"], out_dtype=c["out_dtype"], seed=c["seed"])
    bias = make_bias(case.N, "bf16", seed=540)
    got = run_epi(case, bias, act)
    rows, cols = gi.cell_sample_indices(case.M, case.N, 128, 128, 2, seed=7)
    compare_epi(oracle_lib, case, got, bias, act, rows=rows, cols=cols, what=f"{config} {act}")


@pytest.mark.parametrize("act", ["relu", "gelu", "gelu_tanh"])
def test_activation_accuracy(oracle_lib, act):
    """The GPU's activation functions alone, on a dense grid of exact fp32
    inputs (K == 0, beta == 1, no bias: C = act(C)), against the oracle's fp64
    activations: relative error below 4e-5 (the fp32 evaluation of the fitted
    erfc and of exp, with the conditioning of erfc at large |x|), an absolute
    floor of 1e-36 where results fall into fp32's subnormal range; ReLU exact;
    NaN in, NaN out."""
    import tensor_core_matmul_gb300 as tc
    M, N = 256, 512
    x = np.concatenate([np.linspace(-20.0, 20.0, M * N - 16),
                        [0.0, -0.0, 1e-30, -1e-30, 1e-6, -1e-6, 1e4, -1e4, 88.0, -88.0, 3e38, -3e38,
                         np.inf, -np.inf, np.nan, 1.0]]).astype(np.float32)
    C = torch.from_numpy(x.reshape(N, M)).cuda()
    dummy = torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda")
    tc.gemm_bf16_bias_act(dummy, dummy, C, 1.0, 1.0, activation=act, M=M, N=N, K=0)
    torch.cuda.synchronize()
    got = C.cpu().numpy().reshape(-1).astype(np.float64)
    want = oracle_lib.activation(x.astype(np.float64), act)
    nan_w = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan_w)
    g, w = got[~nan_w], want[~nan_w]
    if act == "relu":
        assert np.array_equal(g, w)
        return
    with np.errstate(invalid="ignore"):  # inf - inf where both are inf (then g == w decides)
        err = np.abs(g - w)
    ok = (err <= 4e-5 * np.abs(w) + 1e-36) | (g == w)
    assert ok.all(), (x[~nan_w][~ok][:5], g[~ok][:5], w[~ok][:5])
