"""GPU parity of the 8-bit-operand GEMM (gemm_fp8: E4M3 or E5M2 inputs, fp32
accumulation on tcgen05 kind::f8f6f4) against the oracle, through the C ABI.
Same rules as the bf16 path (tests/parity.py): fp32 output within
1e-3*sqrt(K)*max(1,|D|); bf16 output within 1 ulp, or the fp32-accumulation
bound where cancellation makes D tiny; integer inputs bit-exact."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import gpu_harness as H
from tests import parity

pytestmark = pytest.mark.gpu

FP8_VARIANTS = [int(v) for v in os.environ.get("FP8_VARIANTS", "0,2,4,5,6,7").split(",")]
FORMATS = ["e4m3", "e5m2"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()


def run_fp8(case: gi.GemmCase, variant: int = 0) -> np.ndarray:
    import tensor_core_matmul_gb300 as tc
    g = H.GuardedC(case)
    tc.gemm_fp8(case.A.cuda(), case.B.cuda(), g.C, case.alpha, case.beta, M=case.M, N=case.N, K=case.K,
                variant=variant)
    torch.cuda.synchronize()
    st, where = tc.check_device_status()
    assert st == 0, f"device status {st} (role {where})"
    g.check_guards()
    return g.result_np()


def compare(o, case: gi.GemmCase, got: np.ndarray, rows=None, cols=None, exact: bool = False, what: str = ""):
    A8, B8, fmt = gi.as_u8(case.A), gi.as_u8(case.B), case.in_format
    if rows is None:
        cols, rows = np.divmod(np.arange(case.M * case.N, dtype=np.int64), case.M)
    D = o.gemm_sampled_f64(case.M, case.N, case.K, A8, B8, rows, cols, H.cin_np(case), case.alpha, case.beta,
                           in_format=fmt)
    g = got[cols, rows]
    if case.out_dtype == gi.OUT_F32:
        if exact:
            parity.check_exact(g, o.round_f32(D), what)
        else:
            parity.check_f32(g, D, case.K, what)
        return
    ref = o.round_bf16(D)
    if exact:
        parity.check_exact(g, ref, what)
        return

    def fallback(flat):
        G = o.absdot_sampled_f64(case.M, case.N, case.K, A8, B8, rows[flat], cols[flat], in_format=fmt)
        return D[flat], abs(case.alpha) * G, case.K
    parity.check_bf16(g, ref, what, fallback=fallback)


@pytest.mark.parametrize("variant", FP8_VARIANTS)
@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16], ids=["f32", "bf16"])
def test_fp8_small_shapes(oracle_lib, variant, fmt, out):
    """Ragged shapes (several tiles, odd and even k-block counts, a K tail
    inside the 128-value k-block), beta on and off."""
    for n, (M, N, K, beta) in enumerate([(200, 300, 320, 0.0), (129, 520, 200, 0.5), (48, 260, 1000, 0.0),
                                         (257, 65, 128, 0.25)]):
        case = gi.make_case(f"f8_{n}", M, N, K, alpha=0.5, beta=beta, out_dtype=out, seed=800 + 10 * n + out,
                            in_format=fmt)
        got = run_fp8(case, variant)
        compare(oracle_lib, case, got, what=f"v{variant} {fmt} {case.name}")


@pytest.mark.parametrize("variant", FP8_VARIANTS)
@pytest.mark.parametrize("fmt", FORMATS)
def test_fp8_integer_exact(oracle_lib, variant, fmt):
    """Integer inputs: every product and partial sum is exact in fp32, so the
    result is bit-exact (fp32 and bf16 output)."""
    for out in (gi.OUT_F32, gi.OUT_BF16):
        case = gi.make_case("f8_int", 300, 270, 700, alpha=1.0, beta=0.5, out_dtype=out, seed=810 + out,
                            kind="integer", in_format=fmt)
        got = run_fp8(case, variant)
        compare(oracle_lib, case, got, exact=True, what=f"v{variant} {fmt} integer")


def test_fp8_padded_leading_dimensions(oracle_lib):
    case = gi.make_case("f8_pad", 131, 77, 300, alpha=1.0, beta=0.0, out_dtype=gi.OUT_F32, seed=820,
                        lda=352, ldb=320, ldc=140, in_format="e4m3")
    compare(oracle_lib, case, run_fp8(case), what="padded")


def test_fp8_stream_k(oracle_lib):
    """Shapes whose plan shares out k-blocks: plain and transposed, repeatable
    bit for bit."""
    import tensor_core_matmul_gb300 as tc
    for n, (M, N, K) in enumerate([(600, 700, 8192), (40, 1000, 16384)]):
        p = tc.plan(M, N, K, 0, torch.cuda.get_device_properties(0).multi_processor_count, in_kind=1)
        assert p["stream_k"] == 1, p
        case = gi.make_case(f"f8_sk{n}", M, N, K, alpha=0.25, beta=0.0, out_dtype=gi.OUT_BF16, seed=830 + n,
                            in_format="e4m3")
        got = run_fp8(case)
        compare(oracle_lib, case, got, what=f"stream-K {case.name}")
        assert np.array_equal(got, run_fp8(case)), "stream-K FP8 not repeatable"


def test_fp8_k_zero(oracle_lib):
    case = gi.make_case("f8_k0", 70, 90, 0, alpha=1.0, beta=0.75, out_dtype=gi.OUT_F32, seed=840, in_format="e5m2")
    compare(oracle_lib, case, run_fp8(case), what="K=0")


@pytest.mark.parametrize("config,fmt", [("s4k", "e4m3"), ("skinny", "e4m3"), ("edge", "e5m2"), ("s8k", "e4m3")])
def test_fp8_full_size_sampled(oracle_lib, config, fmt):
    """The benchmark's workloads with 8-bit operands, in its launch
    configuration, checked at 2 positions in every 128 x 128 cell of C."""
    c = gi.CONFIGS[config]
    case = gi.make_case(config, c["M"], c["N"], c["K"], alpha=c["alpha"], beta=c["beta"], out_dtype=c["out_dtype"],
                        seed=c["seed"], in_format=fmt)
    got = run_fp8(case)
    rows, cols = gi.cell_sample_indices(case.M, case.N, 128, 128, 2, seed=9)
    compare(oracle_lib, case, got, rows=rows, cols=cols, what=f"{config} {fmt}")


def run_fp8_ex(case: gi.GemmCase, variant: int = 0, workspace=None) -> np.ndarray:
    import tensor_core_matmul_gb300 as tc
    g = H.GuardedC(case)
    tc.gemm_fp8_ex(case.A.cuda(), case.B.cuda(), g.C, case.alpha, case.beta, M=case.M, N=case.N, K=case.K,
                   variant=variant, workspace=workspace)
    torch.cuda.synchronize()
    st, where = tc.check_device_status()
    assert st == 0, f"device status {st} (role {where})"
    g.check_guards()
    return g.result_np()


MIXED = [("e4m3", "e5m2"), ("e5m2", "e4m3")]


@pytest.mark.parametrize("variant", FP8_VARIANTS)
@pytest.mark.parametrize("fmts", MIXED, ids=["e4m3xe5m2", "e5m2xe4m3"])
@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16], ids=["f32", "bf16"])
def test_fp8_mixed_formats(oracle_lib, variant, fmts, out):
    """A in one 8-bit format and B in the other (gemm_fp8_ex): ragged shapes
    through every FP8 kernel, the plain and the transposed product (whose
    MMA operands are B and A, so the formats swap places too)."""
    for n, (M, N, K, beta) in enumerate([(200, 300, 320, 0.0), (129, 520, 200, 0.5), (48, 260, 1000, 0.0)]):
        case = gi.make_case(f"f8mix_{n}", M, N, K, alpha=0.5, beta=beta, out_dtype=out, seed=850 + 10 * n + out,
                            in_format=fmts)
        compare(oracle_lib, case, run_fp8_ex(case, variant), what=f"v{variant} {fmts} {case.name}")


@pytest.mark.parametrize("variant", FP8_VARIANTS)
@pytest.mark.parametrize("fmts", MIXED, ids=["e4m3xe5m2", "e5m2xe4m3"])
def test_fp8_mixed_integer_exact(oracle_lib, variant, fmts):
    case = gi.make_case("f8mix_int", 300, 270, 700, alpha=1.0, beta=0.5, out_dtype=gi.OUT_F32, seed=870,
                        kind="integer", in_format=fmts)
    compare(oracle_lib, case, run_fp8_ex(case, variant), exact=True, what=f"v{variant} {fmts} integer")


def test_fp8_caller_workspace(oracle_lib):
    """A stream-K FP8 plan with the caller's workspace equals the library's
    own workspace bit for bit; too small a workspace is refused."""
    import tensor_core_matmul_gb300 as tc
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 600, 700, 8192
    p = tc.plan(M, N, K, 0, sms, in_kind=1)
    assert p["stream_k"] == 1 and p["ws_bytes"] > 0
    case = gi.make_case("f8_ws", M, N, K, alpha=0.5, beta=0.25, out_dtype=gi.OUT_F32, seed=880,
                        in_format=("e4m3", "e5m2"))
    ws = torch.empty(p["ws_bytes"] + 4096, dtype=torch.uint8, device="cuda")
    mine = run_fp8_ex(case, 0, workspace=ws)
    theirs = run_fp8_ex(case, 0)
    assert np.array_equal(mine.view(np.uint32), theirs.view(np.uint32))
    compare(oracle_lib, case, mine, what="fp8 caller workspace")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(tc.TcgemmError):
        run_fp8_ex(case, 0, workspace=small)


@pytest.mark.parametrize("fmt", FORMATS)
def test_fp8_host_buffers(oracle_lib, fmt):
    """gemm_fp8_host on pinned host tensors equals gemm_fp8 on the device bit
    for bit, and the oracle within the usual bound."""
    import tensor_core_matmul_gb300 as tc
    case = gi.make_case(f"f8host_{fmt}", 300, 520, 640, alpha=0.75, beta=0.5, out_dtype=gi.OUT_BF16, seed=890,
                        in_format=fmt)
    C = case.C_in.clone().pin_memory()
    tc.gemm_fp8_host(case.A.pin_memory(), case.B.pin_memory(), C, case.alpha, case.beta, M=case.M, N=case.N,
                     K=case.K)
    torch.cuda.current_stream().synchronize()
    got = C[:, :case.M].contiguous().view(torch.int16).numpy().view(np.uint16)
    dev = run_fp8(case)
    assert np.array_equal(got, dev), "host and device entry points differ"
    compare(oracle_lib, case, got, what=f"fp8 host {fmt}")
