"""GPU tests of the host-buffer entry point (gemm_bf16_host): the library
copies A, B (and C when beta != 0) from host memory, runs the same GEMM as
gemm_bf16 and copies C back.  Its result equals the device entry point's bit
for bit (same kernel, same plan) and the oracle's within the usual bound;
pinned and pageable host buffers, padded leading dimensions and guard bytes
around C on the host."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()


def run_host(case: gi.GemmCase, pinned: bool, stream=None):
    import tensor_core_matmul_gb300 as tc
    A, B = case.A, case.B
    C0 = (case.C_in if case.C_in is not None
          else torch.zeros((case.N, case.ldc), dtype=case.out_torch_dtype()))
    guard = 64
    buf = torch.full((case.N * case.ldc + 2 * guard,), 7, dtype=C0.dtype)
    buf[guard:guard + C0.numel()] = C0.reshape(-1)
    if pinned:
        A, B, buf = A.pin_memory(), B.pin_memory(), buf.pin_memory()
    C = buf[guard:guard + C0.numel()].view(case.N, case.ldc)
    s = torch.cuda.current_stream() if stream is None else stream
    tc.gemm_bf16_host(A, B, C, case.alpha, case.beta, M=case.M, N=case.N, K=case.K, stream=s)
    s.synchronize()
    assert torch.all(buf[:guard] == 7) and torch.all(buf[-guard:] == 7), "write outside C"
    if case.ldc > case.M:
        bits = torch.int16 if C0.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(C[:, case.M:].contiguous().view(bits), C0[:, case.M:].contiguous().view(bits)), \
            "write into the ldc padding"
    got = C[:, :case.M].contiguous()
    return got.view(torch.int16).numpy().view(np.uint16) if got.dtype == torch.bfloat16 else got.numpy()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("M,N,K,out,beta,pad", [(300, 200, 520, gi.OUT_F32, 0.0, 0), (129, 257, 200, gi.OUT_BF16, 0.5, 8),
                                                (130, 100, 96, gi.OUT_F32, 0.0, 8),
                                                (64, 4096, 1024, gi.OUT_BF16, 0.0, 0), (1, 1, 1, gi.OUT_F32, 0.0, 0)])
def test_host_entry_matches_device_entry(oracle_lib, pinned, M, N, K, out, beta, pad):
    case = gi.make_case(f"host{M}", M, N, K, alpha=0.75, beta=beta, out_dtype=out, seed=500 + M,
                        lda=K + pad * 8 if pad else None, ldb=K + pad * 16 if pad else None,
                        ldc=(M + pad * 2 + 7 if out == gi.OUT_BF16 else gi.round_up(M, 4) + 4 * pad) if pad else None)
    got = run_host(case, pinned)
    dev = H.run_case(case, 0).result_np()
    assert np.array_equal(got.view(np.uint8), dev.view(np.uint8)), "host and device entry points differ"
    H.compare_full(oracle_lib, case, got, what=f"host entry {case.name}")


def test_host_entry_two_streams(oracle_lib):
    """Calls on two streams use separate device copies."""
    cases = [gi.make_case(f"hs{i}", 256, 512, 768, alpha=1.0, beta=0.0, out_dtype=gi.OUT_F32, seed=600 + i)
             for i in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    for c, s in zip(cases, streams):
        got = run_host(c, True, s)
        H.compare_full(oracle_lib, c, got, what=c.name)
