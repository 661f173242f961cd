"""GPU parity of the transposed product on CTA pairs (variant 8, M <= 128):
ragged and tiny shapes, every row count the tile height rule can pick,
integer inputs bit-exact, the fused epilogue, and the full-size skinny
workload compared at every element and repeated bit for bit."""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

import gemm_inputs as gi
from tests import gpu_harness as H
from tests import parity

pytestmark = pytest.mark.gpu

PAIR = 8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tensor_core_matmul_gb300 as tc
    tc.lib()


def test_plan_rows_per_cta():
    """r = rows of C's columns per CTA: a multiple of 8 up to 64, one pair
    tile of 2r rows of C^T per resident pair when that fits."""
    import tensor_core_matmul_gb300 as tc
    for M, N in [(64, 8192), (1, 8192), (128, 8192), (40, 9000), (64, 300), (100, 20000)]:
        p = tc.binding.plan_device(M, N, 4096, PAIR)
        assert p["swap"] == 1 and p["cta_group"] == 2 and p["cluster"] == 2
        r = p["arows"]
        assert r % 8 == 0 and 8 <= r <= 64 and p["bm"] == 2 * r
        assert p["tiles_m"] == -(-N // (2 * r)) and p["bn"] == (64 if M <= 64 else 128)
        assert p["stream_k"] == 0 and p["ws_bytes"] == 0


@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16])
def test_small_shape_sweep(oracle_lib, out):
    """Tiny and ragged shapes: every M tail up to 128 rows, N short of, equal
    to and past one pair tile, K below one k-block and with tails."""
    Ms = [1, 7, 33, 64, 65, 100, 128]
    Ns = [1, 15, 16, 17, 129, 300, 1000]
    Ks = [1, 64, 65, 200, 384]
    combos = list(itertools.product(Ms, Ns, Ks))
    rng = np.random.default_rng(8 + out)
    pick = [combos[i] for i in rng.choice(len(combos), size=40, replace=False)]
    pick += [(128, 1000, 384), (1, 1, 1), (64, 16, 64)]
    for n, (M, N, K) in enumerate(pick):
        beta = 0.5 if n % 3 == 0 else 0.0
        case = gi.make_case(f"sp{n}", M, N, K, alpha=1.25, beta=beta, out_dtype=out, seed=800 + n)
        g = H.run_case(case, PAIR)
        H.compare_full(oracle_lib, case, g.result_np(), what=f"pair {M}x{N}x{K} out{out} b{beta}")


@pytest.mark.parametrize("out", [gi.OUT_F32, gi.OUT_BF16])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_integer_bit_exact(oracle_lib, out, beta):
    for n, (M, N, K) in enumerate([(64, 2000, 448), (128, 1500, 1000), (37, 777, 520)]):
        case = gi.make_case(f"spi{n}", M, N, K, alpha=1.0, beta=beta, out_dtype=out, seed=860 + n,
                            kind="integer")
        g = H.run_case(case, PAIR)
        H.compare_full(oracle_lib, case, g.result_np(), exact=True, what=f"pair int {M}x{N}x{K}")


def test_padded_leading_dimensions(oracle_lib):
    case = gi.make_case("sppad", 50, 700, 136, alpha=-2.0, beta=0.25, out_dtype=gi.OUT_F32, seed=870,
                        lda=136 + 24, ldb=136 + 8, ldc=64)
    g = H.run_case(case, PAIR)
    H.compare_full(oracle_lib, case, g.result_np(), what="pair padded ld")


@pytest.mark.parametrize("M,N,K,out", [(64, 8192, 8192, gi.OUT_BF16), (128, 8192, 8192, gi.OUT_BF16),
                                       (100, 8192, 8200, gi.OUT_F32)])
def test_full_size_every_element(oracle_lib, M, N, K, out):
    """The skinny workload's shape (and 128 / 100 rows with a K tail) at full
    size, every element against the oracle, and bit-identical on a repeat."""
    case = gi.make_case(f"spf{M}", M, N, K, alpha=1.0, beta=0.0, out_dtype=out, seed=880 + M)
    got = H.run_case(case, PAIR).result_np()
    stats = H.compare_full(oracle_lib, case, got, what=f"pair full {M}x{N}x{K}")
    H.record_stats(f"pair full {M}x{N}x{K}", stats)
    if out == gi.OUT_BF16:
        assert stats["second_clause"] <= parity.second_clause_cap(K) * stats["size"] + 2, stats
    again = H.run_case(case, PAIR).result_np()
    assert np.array_equal(got.view(np.uint8), again.view(np.uint8))


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_fused_epilogue(oracle_lib, act):
    """bias + activation through the pair kernel equals the same call through
    the single-CTA transposed product (variant 6) bit for bit: both add the
    row's bias and apply the activation to the same fp32 value."""
    import tensor_core_matmul_gb300 as tc
    M, N, K = 48, 3000, 1000
    case = gi.make_case("spe", M, N, K, alpha=0.5, beta=0.0, out_dtype=gi.OUT_BF16, seed=890)
    A, B = case.A.cuda(), case.B.cuda()
    bias = torch.randn(N, generator=torch.Generator().manual_seed(891)).cuda()
    outs = []
    for v in (PAIR, 6):
        C = torch.zeros((N, case.ldc), dtype=torch.bfloat16, device="cuda")
        tc.gemm_bf16_bias_act(A, B, C, case.alpha, 0.0, bias=bias, activation=act, M=M, N=N, K=K, variant=v)
        torch.cuda.synchronize()
        outs.append(C[:, :M].cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_refuses_what_it_does_not_build():
    import tensor_core_matmul_gb300 as tc
    L = tc.lib()
    A = torch.zeros((200, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 208), dtype=torch.float32, device="cuda")
    import ctypes
    st = L.gemm_bf16_variant(200, 64, 64, A.data_ptr(), 64, B.data_ptr(), 64, C.data_ptr(), 208,
                             ctypes.c_float(1.0), ctypes.c_float(0.0), 0, None, PAIR)
    assert st == 1                                   # more than 128 rows of C
