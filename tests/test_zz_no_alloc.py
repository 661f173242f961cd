"""The allocation-free entry point, gemm_bf16_noalloc.

Some callers cannot allocate device memory once they are running: services
with a fixed memory budget decided at start-up, frameworks whose allocator owns
every byte of device memory, and latency-sensitive code that cannot afford the
device-wide synchronisation cudaMalloc may imply.  gemm_bf16 would allocate its
split-K workspace on first use; gemm_bf16_noalloc instead uses a fixed scratch
array compiled into the library and never allocates.

These tests call it through the C ABI and check that it produces what the
regular entry point produces, on two calls in a row (the second call finds the
first call's leftovers in the shared array), and that a shape needing more
scratch than the array holds is refused with a clear error.  The file sorts
last so that a run that stops at the first failure has already run every other
test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()
    return tc


def _run(tc, case, noalloc: bool):
    A, B = case.A.cuda(), case.B.cuda()
    C = (case.C_in.cuda() if case.C_in is not None
         else torch.full((case.N, case.ldc), float("nan"), dtype=case.out_torch_dtype(), device="cuda"))
    stream = torch.cuda.current_stream().cuda_stream
    args = (case.M, case.N, case.K, A.data_ptr(), case.lda, B.data_ptr(), case.ldb, C.data_ptr(), case.ldc,
            case.alpha, case.beta, case.out_dtype, stream, 0)
    st = tc.binding.gemm_bf16_noalloc_raw(*args) if noalloc else tc.gemm_bf16_raw(*args)
    assert st == 0, tc.binding.last_error()
    torch.cuda.synchronize()
    assert tc.check_device_status()[0] == 0
    out = C[:, :case.M].contiguous().cpu()
    if out.dtype == torch.bfloat16:
        return out.view(torch.int16).numpy().view(np.uint16)
    return out.numpy()


def test_noalloc_matches_regular_entry_point_twice(tc):
    """Problems in a row that share out their k-blocks (stream-K), so every
    call uses the scratch array: a pair-tile plan with 20 shared tiles, then
    a single-CTA plan with 64-wide slots (a different slot layout, so stale
    partials of the first call sit where the second writes nothing), then a
    pair-tile plan with 9 shared tiles and another K.  Each result matches
    gemm_bf16 within the fp32 tolerance of the parity tests (and, same plan,
    bit for bit)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for seed, (M, N, K) in [(61, (1024, 1280, 8192)), (62, (128, 4096, 16384)), (63, (600, 700, 12288))]:
        case = gi.make_case(f"noalloc{seed}", M, N, K, alpha=0.75, beta=0.5, out_dtype=gi.OUT_F32,
                            seed=seed)
        need = tc.workspace_bytes(case.M, case.N, case.K, 0, sms)
        assert 0 < need <= tc.binding.noalloc_scratch_bytes()
        got = _run(tc, case, noalloc=True)
        ref = _run(tc, case, noalloc=False)
        parity.check_f32(got, ref.astype(np.float64), case.K, f"noalloc seed {seed}")
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_noalloc_without_split_and_bf16(tc):
    case = gi.make_case("noalloc_plain", 300, 520, 448, alpha=1.0, beta=0.0, out_dtype=gi.OUT_BF16, seed=63)
    got = _run(tc, case, noalloc=True)
    ref = _run(tc, case, noalloc=False)
    parity.check_bf16(got, ref, "noalloc bf16", max_ulp=0)


def test_noalloc_refuses_shapes_beyond_its_scratch(tc):
    """A shape whose plan needs more scratch than the fixed array is refused
    before anything is launched.  (On a 152-SM GB300 every plan fits the
    40 MiB array, and the test says so by skipping.)"""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 896, 2560, 4096
    if tc.workspace_bytes(M, N, K, 1, sms) <= tc.binding.noalloc_scratch_bytes():
        pytest.skip("this device's plan for the shape fits the scratch array")
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((N, M), dtype=torch.float32, device="cuda")
    n0 = tc.launch_count()
    st = tc.binding.gemm_bf16_noalloc_raw(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C.data_ptr(), M, 1.0, 0.0,
                                          gi.OUT_F32, torch.cuda.current_stream().cuda_stream, 1)
    assert st == 1
    assert "scratch" in tc.binding.last_error()
    assert tc.launch_count() == n0
