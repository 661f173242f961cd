"""GPU tests of the autotuner: tcgemm_autotune times the built variants on
the caller's buffers, remembers the fastest, and automatic calls for the same
problem then use it (and still match the oracle)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()
    tc.autotune_clear()
    yield tc
    tc.autotune_clear()


def test_autotune_bf16_then_automatic_calls_use_it(tc, oracle_lib):
    case = gi.make_case("tune", 1000, 1200, 2048, alpha=1.0, beta=0.0, out_dtype=gi.OUT_BF16, seed=1100)
    A, B = case.A.cuda(), case.B.cuda()
    C = torch.empty((case.N, case.ldc), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    v, us = tc.autotune(A, B, C, M=case.M, N=case.N, K=case.K, iters=5, flush=flush)
    assert v in (1, 2, 4, 5, 6, 7) and us > 0
    assert tc.autotune_lookup(case.M, case.N, case.K) == v
    assert tc.check_device_status()[0] == 0
    n0 = tc.launch_count()
    auto = H.run_case(case, 0).result_np()
    explicit = H.run_case(case, v).result_np()
    assert np.array_equal(auto, explicit)  # the automatic call ran the tuned variant
    assert tc.launch_count() > n0
    H.compare_full(oracle_lib, case, auto, what=f"tuned variant {v}")


def test_autotune_fp8_and_layouts_only_pick_built_variants(tc):
    A8 = gi.make_case("t8", 512, 640, 4096, out_dtype=gi.OUT_F32, seed=1101, in_format="e4m3")
    C = torch.empty((A8.N, A8.ldc), dtype=torch.float32, device="cuda")
    v, _ = tc.autotune(A8.A.cuda(), A8.B.cuda(), C, M=A8.M, N=A8.N, K=A8.K, iters=3)
    assert v in (2, 4, 5, 6, 7)
    assert tc.autotune_lookup(A8.M, A8.N, A8.K, in_type=1, out_dtype=0) == v
    base = gi.make_case("tl", 384, 448, 1024, out_dtype=gi.OUT_F32, seed=1102)
    lay = gi.relayout(base, True, True)
    C2 = torch.empty((lay.N, lay.ldc), dtype=torch.float32, device="cuda")
    v2, _ = tc.autotune(lay.A.cuda(), lay.B.cuda(), C2, a_col=True, b_row=True, M=lay.M, N=lay.N, K=lay.K, iters=3)
    assert v2 != 3
    assert tc.autotune_lookup(lay.M, lay.N, lay.K, out_dtype=0, a_col=True, b_row=True) == v2
    tc.autotune_clear()
    assert tc.autotune_lookup(A8.M, A8.N, A8.K, in_type=1, out_dtype=0) == 0
