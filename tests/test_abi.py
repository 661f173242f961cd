"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every symbol the header declares, rejects bad arguments before touching the
device, and its planning / scheduling logic is sound."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tc():
    from tensor_core_matmul_gb300 import _build
    _build.build()
    import tensor_core_matmul_gb300 as tc
    return tc


def header_functions():
    text = open(os.path.join(ROOT, "include", "tcgemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"if", "for", "while", "sizeof"})


def test_exports_every_header_symbol(tc):
    names = header_functions()
    assert "gemm_bf16" in names and len(names) >= 10
    L = ctypes.CDLL(tc.binding.lib_path())
    for n in names:
        assert hasattr(L, n), f"{n} declared in tcgemm.h but not exported"


def test_no_torch_types_in_header():
    text = open(os.path.join(ROOT, "include", "tcgemm.h")).read()
    assert "torch" not in text.lower().replace("pytorch", "") and "at::" not in text


FAKE = 0x10000  # never dereferenced: argument checks run before any CUDA call


@pytest.mark.parametrize("args,status", [
    ((-1, 8, 8, FAKE, 8, FAKE, 8, FAKE, 8), 1),            # negative M
    ((8, 8, 8, FAKE, 4, FAKE, 8, FAKE, 8), 1),             # lda < K
    ((8, 8, 8, FAKE, 8, FAKE, 8, FAKE, 4), 1),             # ldc < M
    ((8, 8, 8, FAKE + 2, 8, FAKE, 8, FAKE * 4, 8), 2),     # A misaligned
    ((8, 8, 12, FAKE, 12, FAKE * 2, 16, FAKE * 4, 8), 2),  # lda*2 not a multiple of 16
    ((6, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE * 4, 6), 2),     # ldc*4 not a multiple of 16
    ((8, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE + 64, 8), 1),    # C overlaps A
    ((8, 8, 8, 0, 8, FAKE, 8, FAKE * 4, 8), 1),            # null A
    ((1 << 31, 8, 8, FAKE, 8, FAKE, 8, FAKE, 1 << 31), 1),  # M too large
])
def test_argument_errors(tc, args, status):
    st = tc.gemm_bf16_raw(*args, 1.0, 0.0, 0, 0)
    assert st == status, (st, tc.binding.last_error())
    assert tc.binding.last_error()


def test_bad_dtype_and_variant(tc):
    assert tc.gemm_bf16_raw(8, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE * 4, 8, 1.0, 0.0, 7, 0) == 1
    assert tc.gemm_bf16_raw(8, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE * 4, 8, 1.0, 0.0, 0, 0, 9) == 1


def test_empty_problems_are_noops(tc):
    assert tc.gemm_bf16_raw(0, 8, 8, 0, 8, 0, 8, 0, 8, 1.0, 0.0, 0, 0) == 0
    assert tc.gemm_bf16_raw(8, 0, 8, 0, 8, 0, 8, 0, 8, 1.0, 0.0, 0, 0) == 0


def test_status_strings(tc):
    L = tc.lib()
    assert L.tcgemm_status_string(0) == b"TCGEMM_OK"
    assert L.tcgemm_status_string(5) == b"TCGEMM_ERR_TIMEOUT"
    assert tc.version() >= 100


@pytest.mark.parametrize("tiles_m,tiles_n,group_m", [(32, 16, 16), (16, 16, 8), (32, 17, 8), (1, 32, 1),
                                                     (5, 3, 4), (64, 32, 16), (7, 1, 2)])
def test_tile_order_is_a_permutation(tc, tiles_m, tiles_n, group_m):
    tm, tn = tc.tile_order(tiles_m, tiles_n, group_m)
    cells = set(zip(tm, tn))
    assert len(cells) == tiles_m * tiles_n
    assert all(0 <= a < tiles_m and 0 <= b < tiles_n for a, b in cells)


def test_tile_order_groups_for_l2(tc):
    """The first `grid` tiles (one wave) stay inside a band of group_m tile rows."""
    tm, tn = tc.tile_order(32, 16, 16, 152)
    assert max(tm) - min(tm) < 16


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (8192, 8192, 8192), (4000, 4100, 4104),
                                   (64, 8192, 8192), (256, 256, 256), (1, 1, 1)])
@pytest.mark.parametrize("variant", [1, 2])
def test_plans(tc, M, N, K, variant):
    p = tc.plan(M, N, K, variant, 152)
    assert p["tiles_m"] * p["bm"] >= M and (p["tiles_m"] - 1) * p["bm"] < M
    assert p["tiles_n"] * p["bn"] >= N and (p["tiles_n"] - 1) * p["bn"] < N
    assert p["num_kb"] * 64 >= K
    assert p["grid"] % p["cta_group"] == 0 and 0 < p["grid"] <= 152
    assert p["grid"] // p["cta_group"] <= p["tiles_m"] * p["tiles_n"]
    assert p["smem"] <= 227 * 1024
