"""GPU parity of the other operand layouts (gemm_bf16_layout: column-major A
and/or row-major B, read by the tensor cores as MN-major operands) against
the oracle's layout-aware definition, through the C ABI.  Same rules as the
bf16 path; integer inputs bit-exact."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import gpu_harness as H
from tests import parity

pytestmark = pytest.mark.gpu

VARIANTS = [int(v) for v in os.environ.get("LAYOUT_VARIANTS", "0,1,2,4,5,6,7").split(",")]
LAYOUTS = [(True, False), (False, True), (True, True)]
IDS = ["NN(A col)", "TT(B row)", "NT(both)"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()


def run_layout(case: gi.GemmCase, variant: int = 0) -> np.ndarray:
    import tensor_core_matmul_gb300 as tc
    g = H.GuardedC(case)
    tc.gemm_bf16_layout(case.A.cuda(), case.B.cuda(), g.C, case.alpha, case.beta, a_col=case.a_col, b_row=case.b_row,
                        M=case.M, N=case.N, K=case.K, variant=variant)
    torch.cuda.synchronize()
    st, where = tc.check_device_status()
    assert st == 0, f"device status {st} (role {where})"
    g.check_guards()
    return g.result_np()


def compare(o, case, got, rows=None, cols=None, exact=False, what=""):
    A, B = gi.as_u16(case.A), gi.as_u16(case.B)
    if rows is None:
        cols, rows = np.divmod(np.arange(case.M * case.N, dtype=np.int64), case.M)
    D = o.gemm_layout_sampled_f64(case.M, case.N, case.K, A, B, case.a_col, case.b_row, rows, cols, H.cin_np(case),
                                  case.alpha, case.beta)
    g = got[cols, rows]
    if case.out_dtype == gi.OUT_F32:
        (parity.check_exact(g, o.round_f32(D), what) if exact else parity.check_f32(g, D, case.K, what))
        return
    ref = o.round_bf16(D)
    if exact:
        parity.check_exact(g, ref, what)
        return

    def fallback(flat):
        G = o.gemm_layout_sampled_f64(case.M, case.N, case.K, A, B, case.a_col, case.b_row, rows[flat], cols[flat],
                                      absolute=True)
        return D[flat], abs(case.alpha) * G, case.K
    parity.check_bf16(g, ref, what, fallback=fallback)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("layout", LAYOUTS, ids=IDS)
@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16], ids=["f32", "bf16"])
def test_layout_small_shapes(oracle_lib, variant, layout, out):
    for n, (M, N, K, beta) in enumerate([(200, 300, 320, 0.0), (129, 520, 200, 0.5), (48, 260, 640, 0.0),
                                         (257, 65, 72, 0.25)]):
        base = gi.make_case(f"lay{n}", M, N, K, alpha=0.5, beta=beta, out_dtype=out, seed=1000 + 10 * n + out)
        case = gi.relayout(base, *layout)
        compare(oracle_lib, case, run_layout(case, variant), what=f"v{variant} {layout} {base.name}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("layout", LAYOUTS, ids=IDS)
def test_layout_integer_exact(oracle_lib, variant, layout):
    base = gi.make_case("lay_int", 300, 270, 500, alpha=1.0, beta=0.5, out_dtype=gi.OUT_F32, seed=1010,
                        kind="integer")
    case = gi.relayout(base, *layout, lda=base.M + 20 if layout[0] else None, ldb=gi.round_up(base.N + 30, 8) if layout[1] else None)
    compare(oracle_lib, case, run_layout(case, variant), exact=True, what=f"v{variant} {layout} integer")


@pytest.mark.parametrize("layout", LAYOUTS, ids=IDS)
def test_layout_stream_k(oracle_lib, layout):
    for n, (M, N, K) in enumerate([(600, 700, 8192), (40, 1000, 8192)]):
        base = gi.make_case(f"lay_sk{n}", M, N, K, alpha=0.25, beta=0.0, out_dtype=gi.OUT_BF16, seed=1020 + n)
        case = gi.relayout(base, *layout)
        got = run_layout(case)
        compare(oracle_lib, case, got, what=f"stream-K {layout} {base.name}")
        assert np.array_equal(got, run_layout(case))


@pytest.mark.parametrize("config,layout", [("s4k", (True, False)), ("s4k", (True, True)), ("edge", (False, True)),
                                           ("skinny", (True, True))])
def test_layout_full_size_sampled(oracle_lib, config, layout):
    case = gi.relayout(gi.config_case(config), *layout)
    got = run_layout(case)
    rows, cols = gi.cell_sample_indices(case.M, case.N, 128, 128, 2, seed=17)
    compare(oracle_lib, case, got, rows=rows, cols=cols, what=f"{config} {layout}")
