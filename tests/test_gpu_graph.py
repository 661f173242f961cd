"""The GEMM entry points inside a CUDA graph: after one ordinary call (which
sets up the library's per-device state and, for stream-K shapes, its
workspace), calls captured on a stream replay with the same results.  Work is
enqueued with plain kernel launches (no host synchronisation, no allocation
after the first call), so a captured sequence of GEMMs replays as one graph
launch."""
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
    return tc


@pytest.mark.parametrize("shape", [(640, 768, 1024), (600, 700, 8192), (48, 2048, 4096)],
                         ids=["tiles", "stream-K", "transposed"])
def test_captured_gemms_replay(tc, oracle_lib, shape):
    M, N, K = shape
    case = gi.make_case("graph", M, N, K, alpha=1.0, beta=0.5, out_dtype=gi.OUT_F32, seed=1200)
    A, B = case.A.cuda(), case.B.cuda()
    C0 = case.C_in.cuda()
    C = C0.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tc.gemm_bf16(A, B, C, case.alpha, case.beta, M=M, N=N, K=K, stream=s)  # set-up outside the capture
    torch.cuda.synchronize()
    eager = C.clone()
    C.copy_(C0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tc.gemm_bf16(A, B, C, case.alpha, case.beta, M=M, N=N, K=K, stream=s)
    for _ in range(2):  # replay twice from the same starting C
        C.copy_(C0)
        g.replay()
        torch.cuda.synchronize()
        assert tc.check_device_status()[0] == 0
        assert torch.equal(C, eager)
    got = C[:, :M].contiguous().cpu().numpy()
    H.compare_full(oracle_lib, case, got, what=f"graph {shape}")
