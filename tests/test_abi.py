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
@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_plans(tc, M, N, K, variant):
    p = tc.plan(M, N, K, variant, 152)
    assert p["tiles_m"] * p["bm"] >= M and (p["tiles_m"] - 1) * p["bm"] < M
    assert p["tiles_n"] * p["bn"] >= N and (p["tiles_n"] - 1) * p["bn"] < N
    assert p["num_kb"] * 64 >= K
    assert p["grid"] % p["cluster"] == 0 and 0 < p["grid"] <= 152
    assert p["grid"] // p["cluster"] <= p["grid_m"] * p["grid_n"] * p["splits"]
    assert p["smem"] <= 227 * 1024


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (8192, 8192, 8192), (4000, 4100, 4104), (64, 8192, 8192),
                                   (1024, 1280, 2048), (513, 200, 1000), (200, 300, 2392), (1, 1, 1),
                                   (129, 257, 65), (100000, 128, 64)])
@pytest.mark.parametrize("variant", [1, 2, 3, 4])
@pytest.mark.parametrize("sms", [152, 148, 20])
def test_split_plan_invariants(tc, M, N, K, variant, sms):
    p = tc.plan(M, N, K, variant, sms)
    tiles = p["grid_m"] * p["grid_n"]
    clusters = sms // p["cluster"]
    assert p["tiles_dp"] + p["tiles_split"] == tiles
    assert p["tiles_dp"] % clusters == 0 or p["tiles_split"] == 0
    if p["tiles_split"] and p["split_n"]:
        assert p["splits"] == 2 and p["tiles_split"] * 2 <= clusters and p["ws_bytes"] == 0
    elif p["tiles_split"]:
        assert p["splits"] >= 2 and p["tiles_split"] * p["splits"] <= clusters
        assert p["splits"] * 4 <= p["num_kb"]
        assert p["ws_bytes"] == 4096 + p["tiles_split"] * p["splits"] * p["cta_group"] * 128 * p["bn"] * 4
        assert p["ws_bytes"] <= 4096 + sms * 128 * 256 * 4
    else:
        assert p["splits"] == 1 and p["ws_bytes"] == 0
    assert tc.workspace_bytes(M, N, K, variant, sms) == p["ws_bytes"]


def test_unit_schedule_covers_every_k_block_once(tc):
    """Simulates the kernel's unit walk on the host for a few plans: every
    (tile, column half, k-block) triple is produced by exactly one cluster."""
    cases = [(4096, 4096, 4096, 2), (8192, 8192, 8192, 2), (1024, 1280, 2048, 2), (64, 8192, 8192, 1),
             (513, 200, 1000, 1), (4000, 4100, 4104, 3), (129, 257, 65, 3), (64, 8192, 8192, 4),
             (4096, 4096, 4096, 1)]
    for (M, N, K, v) in cases:
        p = tc.plan(M, N, K, v, 152)
        G = p["grid"] // p["cluster"]
        seen = {}

        def add(t, half, kb):
            for h in ((0, 1) if half < 0 else (half,)):
                seen[(t, h, kb)] = seen.get((t, h, kb), 0) + 1

        for c in range(G):
            t = c
            while t < p["tiles_dp"]:
                for kb in range(p["num_kb"]):
                    add(t, -1, kb)
                t += G
            if c < p["tiles_split"] * p["splits"]:
                s, piece = divmod(c, p["splits"])
                if p["split_n"]:
                    for kb in range(p["num_kb"]):
                        add(p["tiles_dp"] + s, piece, kb)
                else:
                    kb0 = piece * p["num_kb"] // p["splits"]
                    kb1 = (piece + 1) * p["num_kb"] // p["splits"]
                    assert kb1 > kb0
                    for kb in range(kb0, kb1):
                        add(p["tiles_dp"] + s, -1, kb)
        tiles = p["grid_m"] * p["grid_n"]
        assert len(seen) == tiles * 2 * p["num_kb"] and set(seen.values()) == {1}, (M, N, K, v)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (4000, 4100, 4104), (129, 257, 65), (1, 1, 1)])
def test_multicast_plan_blocks(tc, M, N, K):
    """Variant 3 walks 2 x 2 blocks of 128 x 256 tiles with 4-CTA clusters."""
    p = tc.plan(M, N, K, 3, 152)
    assert p["cluster"] == 4 and p["cta_group"] == 1 and p["bm"] == 128 and p["bn"] == 256
    assert p["grid_m"] == (p["tiles_m"] + 1) // 2 and p["grid_n"] == (p["tiles_n"] + 1) // 2
    assert p["tiles_split"] == 0 and p["ws_bytes"] == 0


def test_auto_variant_choice(tc):
    assert tc.pick_variant(64, 8192, 8192, 152) == 4
    assert tc.pick_variant(128, 4096, 4096, 152) == 4
    assert tc.pick_variant(129, 4096, 4096, 152) == 2
    assert tc.pick_variant(4096, 4096, 4096, 152) == 2
