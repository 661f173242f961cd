"""GPU parity: the CUDA library, called through the C ABI, against the CPU
oracle on the same seeded inputs.

Bars: fp32 output within 1e-3*sqrt(K)*max(1,|ref|); bf16 output within one
bf16 ulp of the oracle's single rounding; integer-valued inputs bit-exact.
Every run also checks guard bands around C and the ldc padding rows, and
with beta == 0 the C buffer is pre-filled with NaN (C must not be read).
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import gpu_harness as H
from tests import parity

pytestmark = pytest.mark.gpu

import os

# 1-CTA, 2-CTA (auto width), narrow 128x64, 2-CTA 256-wide and the two
# transposed-product kernels; TCGEMM_TEST_VARIANTS="1" narrows a run to one.
VARIANTS = [int(v) for v in os.environ.get("TCGEMM_TEST_VARIANTS", "1,2,4,5,6,7").split(",") if v]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()  # fails loudly if the library is missing


@pytest.mark.parametrize("variant", [0] + VARIANTS)
def test_square_256_fp32_full(oracle_lib, variant):
    case = gi.config_case("s256")
    g = H.run_case(case, variant)
    H.compare_full(oracle_lib, case, g.result_np(), what=f"s256 v{variant}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_integer_bit_exact(oracle_lib, variant, out, beta):
    """Integer inputs: every partial sum is an exact integer in fp32, so any
    correct kernel matches the oracle bit for bit (indexing, masks, alpha/beta)."""
    for n, (M, N, K) in enumerate([(300, 520, 448), (129, 257, 65), (513, 200, 1000)]):
        case = gi.make_case(f"int{n}", M, N, K, alpha=1.0, beta=beta, out_dtype=out, seed=40 + n,
                            kind="integer")
        g = H.run_case(case, variant)
        H.compare_full(oracle_lib, case, g.result_np(), exact=True, what=f"int {M}x{N}x{K}")


SWEEP_MN = [1, 7, 64, 65, 127, 129, 257]
SWEEP_K = [1, 16, 63, 64, 65, 192, 384]


@pytest.mark.parametrize("variant", VARIANTS)
def test_small_shape_sweep(oracle_lib, variant):
    """Tiny and ragged shapes, odd and even k-block counts (3 and 6 blocks of
    64), K below one block, every M/N tail."""
    combos = list(itertools.product(SWEEP_MN, SWEEP_MN, SWEEP_K))
    rng = np.random.default_rng(5)
    pick = [combos[i] for i in rng.choice(len(combos), size=60, replace=False)]
    pick += [(1, 1, 1), (257, 257, 384), (7, 129, 65), (129, 7, 63)]
    for n, (M, N, K) in enumerate(pick):
        out = gi.OUT_BF16 if n % 2 else gi.OUT_F32
        beta = 0.5 if n % 3 == 0 else 0.0
        case = gi.make_case(f"sw{n}", M, N, K, alpha=1.5, beta=beta, out_dtype=out, seed=200 + n)
        g = H.run_case(case, variant)
        H.compare_full(oracle_lib, case, g.result_np(), what=f"sweep {M}x{N}x{K} out{out} b{beta}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_padded_leading_dimensions(oracle_lib, variant):
    case = gi.make_case("pad", 200, 300, 136, alpha=-2.0, beta=0.25, out_dtype=gi.OUT_F32, seed=7,
                        lda=136 + 24, ldb=136 + 8, ldc=200 + 12)
    g = H.run_case(case, variant)
    H.compare_full(oracle_lib, case, g.result_np(), what="padded ld")


@pytest.mark.parametrize("name", ["s4k", "s8k", "edge", "skinny"])
def test_configs_full(oracle_lib, name):
    """The full-size workloads in the launch configuration the benchmark times
    (automatic variant), compared with the oracle at every element of C."""
    case = gi.config_case(name)
    g = H.run_case(case, 0)
    got = g.result_np()
    stats = H.compare_full(oracle_lib, case, got, what=name)
    H.record_stats(f"full {name}", stats)
    if case.out_dtype == gi.OUT_BF16:
        assert stats["second_clause"] <= parity.second_clause_cap(case.K) * stats["size"] + 2, stats
    assert not np.isnan(got.astype(np.float32) if got.dtype != np.uint16 else
                        ((got & 0x7FFF) > 0x7F80)).any()


@pytest.mark.parametrize("M,N,K,out,beta", [(128, 8192, 8192, gi.OUT_BF16, 0.0), (100, 8192, 8192, gi.OUT_F32, 0.5),
                                          (40, 9000, 8200, gi.OUT_BF16, 0.0)])
def test_k_split_cluster_sizes_sampled(oracle_lib, M, N, K, out, beta):
    """Skinny shapes the automatic choice gives to the K split over 2-CTA
    clusters (variant 7: 64- and 128-wide tiles of C^T, K tails): sampled at
    2 points of every 128 x 128 cell and along whole rows and columns, and
    repeatable bit for bit."""
    import tensor_core_matmul_gb300 as tc
    assert tc.binding.plan_device(M, N, K, 0)["ks"] == 2
    case = gi.make_case(f"ks{M}", M, N, K, alpha=0.5, beta=beta, out_dtype=out, seed=77 + M)
    got = H.run_case(case, 0).result_np()
    rows, cols = gi.cell_sample_indices(case.M, case.N, 128, 128, 2, seed=21)
    H.compare_sampled(oracle_lib, case, got, rows, cols, what=f"k-split {M}")
    r = np.arange(case.M, dtype=np.int64)
    for j in [0, case.N - 1]:
        H.compare_sampled(oracle_lib, case, got, r, np.full_like(r, j), what=f"k-split {M} col {j}")
    c = np.arange(case.N, dtype=np.int64)
    H.compare_sampled(oracle_lib, case, got, np.full_like(c, case.M - 1), c, what=f"k-split {M} last row")
    again = H.run_case(case, 0).result_np()
    assert np.array_equal(got.view(np.uint8), again.view(np.uint8)), "K split not repeatable"


@pytest.mark.parametrize("name", ["edge", "s8k"])
@pytest.mark.parametrize("variant", VARIANTS)
def test_configs_integer_exact_sampled(oracle_lib, name, variant):
    """The full-size shapes with integer-valued inputs: bit-exact at every
    sampled position for both kernels."""
    case = gi.config_case(name, kind="integer")
    g = H.run_case(case, variant)
    rows, cols = gi.cell_sample_indices(case.M, case.N, 256, 256, 1, seed=12)
    H.compare_sampled(oracle_lib, case, g.result_np(), rows, cols, exact=True, what=f"{name} int")


def test_k_zero_scales_c(oracle_lib):
    case = gi.make_case("k0", 70, 33, 0, alpha=1.0, beta=0.5, out_dtype=gi.OUT_F32, seed=3, kind="integer")
    g = H.run_case(case)
    H.compare_full(oracle_lib, case, g.result_np(), exact=True, what="K=0")
    case0 = gi.make_case("k00", 70, 33, 0, alpha=1.0, beta=0.0, out_dtype=gi.OUT_BF16, seed=3)
    g = H.run_case(case0)
    assert not g.result_np().any()


def test_nonzero_stream_and_repeat(oracle_lib):
    """Runs on a side stream, twice in a row (the second call reuses every
    barrier and TMEM path from a clean start)."""
    case = gi.make_case("st", 384, 640, 320, out_dtype=gi.OUT_BF16, seed=9)
    s = torch.cuda.Stream()
    for _ in range(2):
        with torch.cuda.stream(s):
            g = H.run_case(case, 0, stream=s)
        H.compare_full(oracle_lib, case, g.result_np(), what="stream")


def test_nan_inf_propagate():
    """A NaN in A reaches exactly the outputs of its row; an Inf in B reaches
    exactly the outputs of its column (IEEE propagation, no special casing)."""
    case = gi.make_case("nan", 130, 260, 96, out_dtype=gi.OUT_F32, seed=21)
    A = case.A.clone()
    B = case.B.clone()
    A[5, 17] = float("nan")
    B[200, 3] = float("inf")  # column 200 of B
    case.A, case.B = A, B
    g = H.run_case(case, 0)
    got = g.result_np()  # (N, M)
    assert np.isnan(got[:, 5]).all()
    col = got[200, :]
    assert np.isnan(col[5]) and (~np.isfinite(np.delete(col, 5))).all()
    mask = np.ones_like(got, dtype=bool)
    mask[:, 5] = False
    mask[200, :] = False
    assert np.isfinite(got[mask]).all()


def test_hang_guard_selftest():
    """A wait that nothing satisfies gives up after its limit and reports
    TCGEMM_ERR_TIMEOUT; the context stays usable afterwards."""
    import tensor_core_matmul_gb300 as tc
    st = tc.selftest_timeout(20_000_000)  # 20 ms
    assert st == 5, st
    assert tc.check_device_status()[0] == 0  # status word was cleared
    case = gi.make_case("after", 128, 256, 64, out_dtype=gi.OUT_F32, seed=2, kind="integer")
    H.run_case(case)


@pytest.mark.parametrize("variant", [4, 1, 2])
def test_gemm_gives_up_on_withheld_load(oracle_lib, variant):
    """The GEMM's own hang guard: the producer of CTA 0 withholds its first
    k-block, the MMA thread's wait for it runs out after 20 ms, every role of
    every CTA gives up or finishes, drains its copies and MMAs and exits; the
    call reports TCGEMM_ERR_TIMEOUT within a bounded time, the status word is
    cleared, and the same GEMM run normally afterwards matches the oracle."""
    import time

    import tensor_core_matmul_gb300 as tc
    case = gi.make_case("withheld", 256, 256, 512, alpha=1.0, beta=0.0, out_dtype=gi.OUT_F32, seed=5)
    A, B = case.A.cuda(), case.B.cuda()
    C = torch.zeros((case.N, case.ldc), dtype=torch.float32, device="cuda")
    t0 = time.perf_counter()
    st = tc.binding.selftest_withheld_load(A, B, C, M=case.M, N=case.N, K=case.K, variant=variant,
                                           timeout_ns=20_000_000)
    elapsed = time.perf_counter() - t0
    assert st == 5, (st, tc.binding.last_error())
    assert elapsed < 5.0, elapsed
    assert tc.check_device_status()[0] == 0
    g = H.run_case(case, variant)
    H.compare_full(oracle_lib, case, g.result_np(), what=f"after withheld load v{variant}")


def _split_case():
    # A handful of pair tiles and K = 8192: stream-K shares their k-blocks out
    # over all the pairs.
    return gi.make_case("split", 600, 700, 8192, alpha=0.5, beta=0.25, out_dtype=gi.OUT_F32, seed=31)


def test_split_tiles_repeat_deterministic(oracle_lib):
    """Stream-K tiles: correct, and bit-identical over repeated calls
    (partials are added in K order, whatever order the pieces finish)."""
    import tensor_core_matmul_gb300 as tc
    case = _split_case()
    p = tc.binding.plan_device(case.M, case.N, case.K, 0)
    assert p["stream_k"] == 1 and p["sk_tiles"] > 0, p
    first = None
    for _ in range(3):
        g = H.run_case(case, 0)
        got = g.result_np()
        H.compare_full(oracle_lib, case, got, what="split")
        if first is None:
            first = got
        else:
            assert np.array_equal(got.view(np.uint32), first.view(np.uint32))


def test_caller_workspace_matches_internal(oracle_lib):
    import tensor_core_matmul_gb300 as tc
    case = _split_case()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = tc.workspace_bytes(case.M, case.N, case.K, 0, sms)
    assert need > 0
    ws = torch.full((need + 256,), 0x7F, dtype=torch.uint8, device="cuda")  # no zeroing needed
    A, B = case.A.cuda(), case.B.cuda()
    g = H.GuardedC(case)
    s = torch.cuda.current_stream().cuda_stream
    st = tc.gemm_bf16_ws_raw(case.M, case.N, case.K, A.data_ptr(), case.lda, B.data_ptr(), case.ldb,
                             g.C.data_ptr(), case.ldc, case.alpha, case.beta, case.out_dtype, s, 0,
                             ws.data_ptr(), need)
    assert st == 0, tc.binding.last_error()
    torch.cuda.synchronize()
    g.check_guards()
    ref = H.run_case(case, 0).result_np()
    assert np.array_equal(g.result_np().view(np.uint32), ref.view(np.uint32))
    st = tc.gemm_bf16_ws_raw(case.M, case.N, case.K, A.data_ptr(), case.lda, B.data_ptr(), case.ldb,
                             g.C.data_ptr(), case.ldc, case.alpha, case.beta, case.out_dtype, s, 0,
                             ws.data_ptr(), need - 1)
    assert st == 1


@pytest.mark.parametrize("variant", VARIANTS)
def test_split_small_k_pieces(oracle_lib, variant):
    """Few tiles and a long K: maximal splitting, with pieces of uneven length."""
    case = gi.make_case("longk", 200, 300, 64 * 37 + 24, alpha=1.0, beta=0.0, out_dtype=gi.OUT_BF16, seed=33)
    g = H.run_case(case, variant)
    H.compare_full(oracle_lib, case, g.result_np(), what=f"long K v{variant}")


@pytest.mark.parametrize("variant", [1, 2, 4, 5, 6])
@pytest.mark.parametrize("kind", ["integer", "normal"])
def test_stream_k_small_problems(oracle_lib, variant, kind):
    """Few tiles and a long K, so stream-K shares every k-block out over all
    clusters (ragged edges, K not a multiple of 64): integer inputs bit-exact,
    N(0,1) inputs within tolerance, beta = 0.5 over C."""
    import tensor_core_matmul_gb300 as tc
    bm = {1: 128, 2: 256, 4: 128, 5: 256, 6: 64}[variant]
    bn = {1: 256, 2: 256, 4: 64, 5: 256, 6: 128}[variant]
    shapes = [(bm * 2 - 40, bn * 3 - 24, 8000), (bm - 7, bn * 5 - 100, 12000)]
    for n, (M, N, K) in enumerate(shapes):
        p = tc.binding.plan_device(M, N, K, variant)
        assert p["stream_k"] == 1, (M, N, K, p)
        case = gi.make_case("sk", M, N, K, alpha=1.0, beta=0.5, out_dtype=gi.OUT_F32 if n == 0 else gi.OUT_BF16,
                            seed=70 + n, kind=kind)
        g = H.run_case(case, variant)
        H.compare_full(oracle_lib, case, g.result_np(), exact=(kind == "integer"), what=f"stream-K v{variant} {M}x{N}x{K}")


def test_device_plan_and_width_choice():
    import tensor_core_matmul_gb300 as tc
    info = tc.binding.device_info()
    assert info["sms"] >= 100 and 0 < info["max_pairs"] <= info["sms"] // 2
    p = tc.binding.plan_device(4096, 4096, 4096, 0)
    assert p["cta_group"] == 2 and p["bn"] in (224, 256)
    assert p["grid"] == 2 * min(info["max_pairs"], p["tiles_m"] * p["tiles_n"])
    assert tc.binding.plan_device(64, 8192, 8192, 0)["swap"] == 1
    assert tc.binding.plan_device(100, 8192, 8192, 0)["arows"] == 128
