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


@pytest.mark.parametrize("args,out,status", [
    ((8, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE * 4, 8), 2, 1),   # int8 output is not offered on host buffers
    ((8, 8, 8, FAKE, 4, FAKE * 2, 8, FAKE * 4, 8), 0, 1),   # lda < K
    ((8, 8, 8, FAKE + 2, 8, FAKE * 2, 8, FAKE * 4, 8), 0, 2),  # A misaligned
    ((8, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE + 64, 8), 0, 1),  # C overlaps A
    ((8, 8, 8, FAKE, 8, 0, 8, FAKE * 4, 8), 0, 1),          # null B
])
def test_host_entry_argument_errors(tc, args, out, status):
    """The host-buffer entry point checks its arguments before any CUDA call."""
    st = tc.binding.gemm_bf16_host_raw(*args, 1.0, 0.0, out, 0)
    assert st == status, (st, tc.binding.last_error())
    assert tc.binding.last_error()


def test_host_entry_empty_is_noop(tc):
    assert tc.binding.gemm_bf16_host_raw(0, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE * 4, 8, 1.0, 0.0, 0, 0) == 0


def test_bad_dtype_and_variant(tc):
    assert tc.gemm_bf16_raw(8, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE * 4, 8, 1.0, 0.0, 7, 0) == 1
    assert tc.gemm_bf16_raw(8, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE * 4, 8, 1.0, 0.0, 0, 0, 9) == 1


@pytest.mark.parametrize("bias,bias_dtype,act,status", [
    (None, 0, 4, 1),               # unknown activation
    (None, 0, -1, 1),              # unknown activation
    (FAKE * 8, 3, 0, 1),           # unknown bias dtype
    (None, 1, 0, 1),               # bias dtype given, pointer NULL
    (FAKE * 8, 0, 0, 1),           # pointer given with TCGEMM_BIAS_NONE
    (FAKE * 8 + 2, 1, 1, 2),       # fp32 bias not 4-byte aligned
    (FAKE * 8 + 1, 2, 2, 2),       # bf16 bias not 2-byte aligned
    (FAKE * 4 + 8, 1, 0, 1),       # bias overlaps C
])
def test_epilogue_argument_errors(tc, bias, bias_dtype, act, status):
    """The fused-epilogue entry point checks its extra arguments on the host,
    before anything is launched (C is at FAKE*4, 8 x 8 fp32)."""
    st = tc.binding.gemm_bf16_bias_act_raw(8, 8, 8, FAKE, 8, FAKE * 2, 8, FAKE * 4, 8, 1.0, 0.0, 0, bias,
                                           bias_dtype, act, 0, 0)
    assert st == status, (st, tc.binding.last_error())
    assert tc.binding.last_error()


@pytest.mark.parametrize("args,fmt,variant,status", [
    ((8, 8, 16, FAKE, 16, FAKE * 2, 16, FAKE * 4, 8), 2, 0, 1),     # unknown FP8 format
    ((8, 8, 16, FAKE, 16, FAKE * 2, 16, FAKE * 4, 8), 0, 1, 1),     # variant not built for FP8
    ((8, 8, 16, FAKE, 16, FAKE * 2, 16, FAKE * 4, 8), 1, 3, 1),     # 3 names no kernel
    ((8, 8, 8, FAKE, 8, FAKE * 2, 16, FAKE * 4, 8), 0, 0, 2),       # lda = 8 bytes: not a 16-byte multiple
    ((8, 8, 16, FAKE + 8, 16, FAKE * 2, 16, FAKE * 4, 8), 1, 0, 2), # A misaligned
])
def test_fp8_argument_errors(tc, args, fmt, variant, status):
    st = tc.binding.gemm_fp8_raw(*args, 1.0, 0.0, 0, fmt, 0, variant)
    assert st == status, (st, tc.binding.last_error())


@pytest.mark.parametrize("fa,fb,status", [(2, 0, 1), (0, 2, 1), (-1, 1, 1), (1, 7, 1)])
def test_fp8_ex_argument_errors(tc, fa, fb, status):
    """gemm_fp8_ex checks each operand's format on the host."""
    st = tc.lib().gemm_fp8_ex(8, 8, 16, FAKE, 16, fa, FAKE * 2, 16, fb, FAKE * 4, 8, 1.0, 0.0, 0, None, 0, None, 0)
    assert st == status, (st, tc.binding.last_error())
    assert b"FP8 format" in tc.lib().tcgemm_last_error()


def test_fp8_host_argument_errors(tc):
    L = tc.lib()
    assert L.gemm_fp8_host(8, 8, 16, FAKE, 16, FAKE * 2, 16, FAKE * 4, 8, 1.0, 0.0, 0, 5, None) == 1
    assert L.gemm_fp8_host(8, 8, 16, FAKE, 16, FAKE * 2, 16, FAKE * 4, 8, 1.0, 0.0, 2, 0, None) == 1   # int8 out


@pytest.mark.parametrize("in_type,scale,variant,status", [
    (3, FAKE * 16, 0, 1),          # unknown operand type
    (0, None, 0, 1),               # no row scales
    (1, FAKE * 16 + 4, 0, 2),      # row scales not 16-byte aligned
    (0, FAKE * 16, 1, 1),          # variant not built for int8 output
    (2, FAKE * 4, 0, 1),           # row scales overlap Q (Q at FAKE*4, 16 x 8 int8)
])
def test_quant_argument_errors(tc, in_type, scale, variant, status):
    st = tc.binding.gemm_quant_i8_raw(16, 8, 16, FAKE, 16, FAKE * 2, 16, in_type, FAKE * 4, 16, 1.0, None, 0, 0,
                                      scale, 0, 0, variant)
    assert st == status, (st, tc.binding.last_error())


@pytest.mark.parametrize("args,status", [
    ((8, 8, 16, FAKE, 16, 2, FAKE * 2, 16, 1), 1),      # unknown A layout
    ((8, 8, 16, FAKE, 4, 1, FAKE * 2, 16, 1), 1),       # column-major A: lda < M
    ((8, 12, 16, FAKE, 16, 0, FAKE * 2, 8, 0), 1),      # row-major B: ldb < N
    ((8, 8, 16, FAKE, 12, 1, FAKE * 2, 16, 1), 2),      # lda*2 not a multiple of 16
])
def test_layout_argument_errors(tc, args, status):
    st = tc.binding.gemm_bf16_layout_raw(*args, FAKE * 4, 8, 1.0, 0.0, 0, 0, 0)
    assert st == status, (st, tc.binding.last_error())


def test_row_major_b_takes_256_wide_pairs(tc):
    assert tc.plan(4096, 4096, 4096, 0, 152)["bn"] == 224
    assert tc.plan(4096, 4096, 4096, 0, 152, b_row=True)["bn"] == 256
    assert tc.plan(4096, 4096, 4096, 0, 152, a_col=True)["bn"] == 224


def test_variant_number_3_names_no_kernel(tc):
    """Variant number 3 is unused: every entry point refuses it on the host,
    and no plan exists for it."""
    assert tc.binding.gemm_bf16_layout_raw(8, 8, 16, FAKE, 8, 1, FAKE * 2, 16, 1, FAKE * 4, 8, 1.0, 0.0, 0, 0,
                                           3) == 1
    assert tc.lib().gemm_bf16_variant(8, 8, 16, FAKE, 16, FAKE * 2, 16, FAKE * 4, 8, ctypes.c_float(1.0),
                                      ctypes.c_float(0.0), 0, None, 3) == 1
    assert b"unknown variant" in tc.lib().tcgemm_last_error()
    with pytest.raises(tc.TcgemmError):
        tc.plan(4096, 4096, 4096, 3, 152)


def test_autotune_table_starts_empty_and_rejects_bad_arguments(tc):
    tc.autotune_clear()
    assert tc.autotune_lookup(4096, 4096, 4096) == 0
    best = ctypes.c_int(-1)
    L = tc.lib()
    assert L.tcgemm_autotune(8, 8, 16, FAKE, 16, 0, FAKE * 2, 16, 1, 0, FAKE * 4, 8, 1.0, 0.0, 0, 0, None, 0, None,
                             ctypes.byref(best), None) == 1          # iters = 0
    assert L.tcgemm_autotune(8, 8, 16, FAKE, 16, 0, FAKE * 2, 16, 1, 0, FAKE * 4, 8, 1.0, 0.0, 2, 5, None, 0, None,
                             ctypes.byref(best), None) == 1          # int8 output is not tuned
    assert L.tcgemm_autotune(8, 8, 16, FAKE, 16, 0, FAKE * 2, 16, 1, 0, FAKE * 4, 8, 1.0, 0.0, 0, 5, None, 64, None,
                             ctypes.byref(best), None) == 1          # flush size without a buffer
    assert best.value == -1


def test_int8_output_needs_the_quantising_entry_point(tc):
    assert tc.gemm_bf16_raw(16, 8, 16, FAKE, 16, FAKE * 2, 16, FAKE * 4, 16, 1.0, 0.0, 2, 0) == 1
    assert "scale" in tc.binding.last_error()


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (64, 8192, 8192), (600, 700, 8192), (600, 700, 4096)])
def test_fp8_plans_count_128_value_k_blocks(tc, M, N, K):
    p8 = tc.plan(M, N, K, 0, 152, in_kind=1)
    p16 = tc.plan(M, N, K, 0, 152)
    assert p8["num_kb"] == (K + 127) // 128 and p16["num_kb"] == (K + 63) // 64
    assert p8["smem"] == p16["smem"] or p8["bn"] != p16["bn"]


def test_epilogue_empty_problem_is_noop(tc):
    assert tc.binding.gemm_bf16_bias_act_raw(0, 8, 8, 0, 8, 0, 8, 0, 8, 1.0, 0.0, 0, FAKE, 1, 2, 0, 0) == 0


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


def _hilbert_reference(k: int):
    """Cells of the 2^k x 2^k Hilbert curve by the recursive construction
    (each square split into four quarter-squares traversed with their axes
    exchanged, unchanged, unchanged, and reversed-exchanged), an
    independent restatement of the curve, started along the second axis."""
    out = []

    def rec(x0, y0, xi, xj, yi, yj, n):
        if n == 0:
            out.append((int(x0 + (xi + yi) / 2), int(y0 + (xj + yj) / 2)))
            return
        rec(x0, y0, yi / 2, yj / 2, xi / 2, xj / 2, n - 1)
        rec(x0 + xi / 2, y0 + xj / 2, xi / 2, xj / 2, yi / 2, yj / 2, n - 1)
        rec(x0 + xi / 2 + yi / 2, y0 + xj / 2 + yj / 2, xi / 2, xj / 2, yi / 2, yj / 2, n - 1)
        rec(x0 + xi / 2 + yi, y0 + xj / 2 + yj, -yi / 2, -yj / 2, -xi / 2, -xj / 2, n - 1)

    s = 2 ** k
    rec(0.0, 0.0, 0.0, float(s), float(s), 0.0, k)
    return out


@pytest.mark.parametrize("tiles_m,tiles_n", [(1, 1), (2, 2), (4, 4), (32, 32), (16, 19), (16, 17), (19, 16),
                                             (5, 3), (1, 32), (33, 2), (64, 64), (7, 100)])
def test_hilbert_order_matches_recursive_curve(tc, tiles_m, tiles_n):
    """The Hilbert visiting order (host copy of the device function) is the
    recursive curve of the enclosing power-of-two square with the cells
    outside the grid dropped: a permutation of the grid, and on full squares
    every step moves to a neighbouring tile."""
    tm, tn = tc.tile_order_hilbert(tiles_m, tiles_n)
    k = max(0, (max(tiles_m, tiles_n) - 1).bit_length())
    ref = [(x, y) for x, y in _hilbert_reference(k) if x < tiles_m and y < tiles_n]
    assert list(zip(tm, tn)) == ref
    assert len(set(ref)) == tiles_m * tiles_n
    if tiles_m == tiles_n and tiles_m & (tiles_m - 1) == 0:
        assert all(abs(a - c) + abs(b - d) == 1 for (a, b), (c, d) in zip(ref, ref[1:]))


def test_hilbert_rounds_are_compact(tc):
    """A round of 76 pair tiles on the 32 x 32 grid of 8192^3 covers a patch
    no larger than the grouped order's, and consecutive rounds share edges."""
    tm, tn = tc.tile_order_hilbert(32, 32)
    for r in range(1024 // 76):
        cells = list(zip(tm[76 * r:76 * (r + 1)], tn[76 * r:76 * (r + 1)]))
        rows = len({a for a, _ in cells})
        cols = len({b for _, b in cells})
        assert rows * cols <= 2 * 76 + 64, (r, rows, cols)
    with pytest.raises(tc.TcgemmError):
        tc.tile_order_hilbert(4, 4, 17)


def test_tile_order_groups_for_l2(tc):
    """The first `grid` tiles (one wave) stay inside a band of group_m tile rows."""
    tm, tn = tc.tile_order(32, 16, 16, 152)
    assert max(tm) - min(tm) < 16


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (8192, 8192, 8192), (4000, 4100, 4104),
                                   (64, 8192, 8192), (256, 256, 256), (1, 1, 1)])
@pytest.mark.parametrize("variant", [1, 2, 4, 5, 6, 7])
def test_plans(tc, M, N, K, variant):
    p = tc.plan(M, N, K, variant, 152)
    if p["swap"]:
        M, N = N, M          # the launch describes C^T
    assert p["tiles_m"] * p["bm"] >= M and (p["tiles_m"] - 1) * p["bm"] < M
    assert p["tiles_n"] * p["bn"] >= N and (p["tiles_n"] - 1) * p["bn"] < N
    assert p["num_kb"] * 64 >= K
    assert p["grid"] % p["cluster"] == 0 and 0 < p["grid"] <= 152
    assert p["grid"] // p["cluster"] <= p["grid_m"] * p["grid_n"] or p["stream_k"]
    assert p["smem"] <= 227 * 1024


SK_SHAPES = [(4096, 4096, 4096), (8192, 8192, 8192), (4000, 4100, 4104), (64, 8192, 8192), (512, 512, 16384),
             (513, 200, 1000), (200, 300, 2392), (1, 1, 1), (129, 257, 65), (100000, 128, 64), (3000, 5000, 777)]


@pytest.mark.parametrize("M,N,K", SK_SHAPES)
@pytest.mark.parametrize("variant", [1, 2, 4, 5, 6, 7])
@pytest.mark.parametrize("sms", [152, 148, 20])
def test_stream_k_plan_invariants(tc, M, N, K, variant, sms):
    p = tc.plan(M, N, K, variant, sms)
    units = p["grid_m"] * p["grid_n"]
    clusters = p["grid"] // p["cluster"]
    assert p["tiles_dp"] + p["sk_tiles"] == units
    if p["stream_k"]:
        full = (sms // p["cluster"]) if p["cluster"] > 1 else sms
        assert clusters == min(full, sms // p["cluster"]) and p["tiles_dp"] % clusters == 0
        assert 0 < p["sk_tiles"] < clusters and 2 * p["sk_tiles"] <= clusters and p["tiles_dp"] == 0
        assert p["sk_iters"] == p["sk_tiles"] * p["num_kb"] >= 4 * clusters
        assert p["ws_bytes"] == 2 * clusters * p["cta_group"] * 128 * p["bn"] * 4
        assert p["ws_bytes"] <= 2 * sms * 128 * 256 * 4
    else:
        assert p["sk_tiles"] == 0 and p["ws_bytes"] == 0
    assert tc.workspace_bytes(M, N, K, variant, sms) == p["ws_bytes"]


def _sk_slot(c, t_begin, iters, clusters):
    # the fixup's formula, restated: a cluster's first segment uses slot 2c
    return 2 * c + (0 if (c * iters) // clusters >= t_begin else 1)


@pytest.mark.parametrize("M,N,K,v", [(4096, 4096, 4096, 2), (8192, 8192, 8192, 2), (512, 512, 16384, 2),
                                     (256, 2048, 8192, 1), (600, 700, 8192, 5), (1024, 1280, 2048, 2),
                                     (64, 8192, 8192, 1), (513, 200, 1000, 1), (4000, 4100, 4104, 4),
                                     (129, 257, 65, 7), (64, 8192, 8192, 4), (4096, 4096, 4096, 1),
                                     (4096, 4096, 4096, 5), (8192, 8192, 8192, 5), (4000, 4100, 4104, 2),
                                     (200, 300, 2392, 2), (3000, 5000, 777, 2), (64, 8192, 8192, 6),
                                     (50, 3000, 5000, 6)])
def test_unit_schedule_covers_every_k_block_once(tc, M, N, K, v):
    """Runs the kernel's own unit iterator (host copy) for every cluster:
    every (tile, k-block) is produced exactly once; the pieces of each
    stream-K tile are numbered 0..n-1 in K order, agree on n, use distinct
    workspace slots, and the slot the fixup computes for piece i is the slot
    that piece writes."""
    p = tc.plan(M, N, K, v, 152)
    G = p["grid"] // p["cluster"]
    seen = {}
    pieces = {}
    for c in range(G):
        for u in tc.binding.units(M, N, K, v, 152, c):
            assert 0 <= u["kb0"] < u["kb1"] <= p["num_kb"]
            for kb in range(u["kb0"], u["kb1"]):
                seen[(u["tile"], kb)] = seen.get((u["tile"], kb), 0) + 1
            if u["slot"] >= 0:
                pieces.setdefault(u["sk_tile"], []).append((u["kb0"], u["piece"], u["npieces"], u["slot"], c))
            else:
                assert u["kb0"] == 0 and u["kb1"] == p["num_kb"]
    assert len(seen) == p["grid_m"] * p["grid_n"] * p["num_kb"] and set(seen.values()) == {1}
    slots = set()
    for t, ps in pieces.items():
        ps.sort()
        n = ps[0][2]
        assert [x[1] for x in ps] == list(range(n)) and all(x[2] == n for x in ps) and n >= 2
        first = ps[0][4]
        for i, (_, _, _, slot, c) in enumerate(ps):
            assert c == first + i
            assert slot == _sk_slot(c, t * p["num_kb"], p["sk_iters"], G)
            assert slot not in slots
            slots.add(slot)
    assert all(0 <= sl < 2 * G for sl in slots)


def test_width_choice(tc):
    """The pair kernel takes 224-wide tiles where whole rounds of them finish
    sooner (4096^2: 304 tiles = 4 rounds instead of 256 tiles = 3.4 rounds);
    variant 5 always uses 256; skinny shapes load 64-row A tiles; stream-K only
    for problems with at most half a round of tiles and a long K."""
    assert tc.plan(4096, 4096, 4096, 2, 152)["bn"] == 224    # 304 tiles = 4 full rounds of 76 pairs
    assert tc.plan(8192, 8192, 8192, 2, 152)["bn"] == 256
    assert tc.plan(4096, 4096, 4096, 5, 152)["bn"] == 256
    assert tc.plan(64, 8192, 8192, 4, 152)["arows"] == 64
    assert tc.plan(128, 8192, 8192, 4, 152)["arows"] == 128
    assert tc.plan(64, 8192, 8192, 0, 152)["swap"] == 1
    assert tc.plan(4096, 4096, 4096, 2, 152)["stream_k"] == 0
    assert tc.plan(1024, 1280, 2048, 2, 152)["stream_k"] == 0   # K too short to pay for it
    assert tc.plan(512, 512, 16384, 2, 152)["stream_k"] == 1    # 4 tiles, long K


def test_k_split_plan(tc):
    """Variant 7: the transposed product with each tile's k-blocks split over
    a 2-CTA cluster: two CTAs per tile, no stream-K, no workspace; a single
    k-block cannot be split and runs on one CTA per tile."""
    p = tc.plan(64, 8192, 8192, 7, 152)
    assert (p["swap"], p["ks"], p["cluster"], p["grid"], p["stream_k"], p["ws_bytes"]) == (1, 2, 2, 128, 0, 0)
    assert p["tiles_m"] == 64 and p["tiles_n"] == 1 and p["bn"] == 64
    p = tc.plan(40, 30000, 640, 7, 152)      # 235 tiles: rounds of 76 clusters
    assert p["ks"] == 2 and p["grid"] == 152 and p["stream_k"] == 0
    p = tc.plan(64, 8192, 64, 7, 152)
    assert p["ks"] == 1 and p["cluster"] == 1 and p["bn"] == 64
    p = tc.plan(128, 8192, 8192, 7, 152)      # 64 < M <= 128: 128 x 128 tiles of C^T
    assert (p["ks"], p["bn"], p["grid"], p["tiles_n"]) == (2, 128, 128, 1) and p["smem"] <= 227 * 1024
    p = tc.plan(300, 200, 320, 7, 152)        # C^T is 200 x 300: 2 x 3 tiles of 128 x 128
    assert (p["ks"], p["bn"], p["tiles_m"], p["tiles_n"]) == (2, 128, 2, 3)
    assert tc.plan(64, 8192, 8192, 6, 152)["ks"] == 1


@pytest.mark.parametrize("M,N,K", [(64, 8192, 8192), (1, 1, 1), (128, 8192, 8192), (100, 20000, 640),
                                   (40, 9000, 8200), (64, 16, 64)])
@pytest.mark.parametrize("sms", [152, 148, 20])
def test_swap_pair_plan(tc, M, N, K, sms):
    """Variant 8: C^T on CTA pairs, r = rows of C^T per CTA (a multiple of 8,
    at most 64) so that the 2r-row pair tiles cover C^T with about one tile
    per resident pair; whole K per pair, no stream-K, no workspace."""
    p = tc.plan(M, N, K, 8, sms)
    r = p["arows"]
    assert (p["swap"], p["cta_group"], p["cluster"], p["ks"], p["stream_k"], p["ws_bytes"]) == (1, 2, 2, 1, 0, 0)
    assert r % 8 == 0 and 8 <= r <= 64 and p["bm"] == 2 * r
    assert p["tiles_m"] == -(-N // (2 * r)) and p["tiles_n"] == 1 and p["bn"] == (64 if M <= 64 else 128)
    pairs = sms // 2
    if r < 64:
        assert p["tiles_m"] <= pairs                      # one tile per pair at most
        assert r == 8 or -(-N // (2 * (r - 8))) > pairs   # and r is the smallest that fits
    assert p["grid"] == 2 * min(p["tiles_m"], pairs) and p["smem"] <= 227 * 1024
    assert p["num_kb"] == -(-K // 64)


def test_swap_pair_refusals(tc):
    for kwargs in [dict(M=129, N=1000, K=64), dict(M=64, N=1000, K=64, a_col=True),
                   dict(M=64, N=1000, K=64, in_kind=1)]:
        with pytest.raises(tc.TcgemmError):
            tc.plan(kwargs.pop("M"), kwargs.pop("N"), kwargs.pop("K"), 8, 152, **kwargs)
    with pytest.raises(tc.TcgemmError):
        tc.binding.autotune_set(256, 64, 256, 8)          # more than 128 rows of C
    with pytest.raises(tc.TcgemmError):
        tc.binding.autotune_set(64, 4096, 256, 8, in_type=1)


def test_withheld_load_selftest_argument_errors(tc):
    """The GEMM give-up self test checks its arguments on the host: only the
    plain-product variants, positive sizes, a limit in (0, 10 s]."""
    L = tc.lib()
    args = (256, 256, 512, FAKE, 512, FAKE * 2, 512, FAKE * 4, 256)
    assert L.tcgemm_selftest_withheld_load(*args, 6, 20_000_000, None) == 1
    assert L.tcgemm_selftest_withheld_load(*args, 3, 20_000_000, None) == 1
    assert L.tcgemm_selftest_withheld_load(*args, 2, 0, None) == 1
    assert L.tcgemm_selftest_withheld_load(*args, 2, 11_000_000_000, None) == 1
    assert L.tcgemm_selftest_withheld_load(0, 256, 512, FAKE, 512, FAKE * 2, 512, FAKE * 4, 256, 2,
                                           20_000_000, None) == 1


def test_noalloc_fit_decision(tc):
    """The test gemm_bf16_noalloc applies before launching: a plan fits its
    fixed scratch array when its workspace does.  Every plan of a 152-SM
    GB300 fits (2 slots x 76 pairs x 256 KiB = 38 MiB of 40); on a device
    with 256 SMs a stream-K pair plan needs 64 MiB and is refused."""
    b = tc.binding
    cap = b.noalloc_scratch_bytes()
    for M, N, K, v in [(600, 700, 8192, 0), (896, 2560, 4096, 1), (128, 4096, 16384, 0), (4096, 4096, 4096, 0)]:
        need = tc.workspace_bytes(M, N, K, v, 152)
        assert b.noalloc_fits(M, N, K, v, 152) == (need <= cap) is True
    assert tc.workspace_bytes(600, 700, 8192, 0, 256) > cap
    assert b.noalloc_fits(600, 700, 8192, 0, 256) is False
    assert b.noalloc_fits(896, 2560, 4096, 1, 256) is False
    assert b.noalloc_fits(4096, 4096, 4096, 0, 256) is True        # no split: no scratch needed
    with pytest.raises(tc.TcgemmError):
        b.noalloc_fits(0, 1, 1, 0, 152)


def test_auto_variant_choice(tc):
    assert tc.pick_variant(64, 8192, 8192, 152) == 7      # 64 tiles: 128 of 152 SMs, K split in halves
    assert tc.pick_variant(64, 4096, 8192, 152) == 6      # 32 tiles: stream-K over all SMs instead
    assert tc.pick_variant(64, 8192, 256, 152) == 6       # 4 k-blocks: too short to split
    assert tc.pick_variant(64, 12288, 8192, 152) == 6     # 96 tiles: more than a round of clusters
    assert tc.pick_variant(128, 8192, 8192, 152) == 7     # 128-wide tiles of C^T, K split
    assert tc.pick_variant(100, 8192, 8192, 152) == 7
    assert tc.pick_variant(128, 12288, 8192, 152) == 4
    assert tc.pick_variant(128, 4096, 4096, 152) == 4
    assert tc.pick_variant(64, 128, 4096, 152) == 4
    assert tc.pick_variant(129, 4096, 4096, 152) == 2
    assert tc.pick_variant(4096, 4096, 4096, 152) == 2


def test_autotune_table_set_save_load(tc, tmp_path):
    """The tuned-choice table: a choice set by hand is what an automatic call
    would use (lookup), survives a save / clear / load round trip, and a
    variant not built for the problem is refused.  No GPU needed."""
    b = tc.binding
    b.autotune_clear()
    b.autotune_set(1000, 1200, 2048, 5)
    b.autotune_set(512, 640, 4096, 4, in_type=1, out_dtype=0)
    b.autotune_set(384, 448, 1024, 2, out_dtype=0, a_col=True, b_row=True, beta_nonzero=True)
    assert b.autotune_lookup(1000, 1200, 2048) == 5
    assert b.autotune_lookup(512, 640, 4096, in_type=1, out_dtype=0) == 4
    assert b.autotune_lookup(512, 640, 4096, in_type=2, out_dtype=0) == 0   # E5M2 is another problem
    path = tmp_path / "tuned.txt"
    assert b.autotune_save(path) == 3
    b.autotune_clear()
    assert b.autotune_lookup(1000, 1200, 2048) == 0
    assert b.autotune_load(path) == 3
    assert b.autotune_lookup(1000, 1200, 2048) == 5
    assert b.autotune_lookup(384, 448, 1024, out_dtype=0, a_col=True, b_row=True, beta_nonzero=True) == 2
    b.autotune_set(1000, 1200, 2048, 0)                                      # variant 0 removes the choice
    assert b.autotune_lookup(1000, 1200, 2048) == 0
    b.autotune_clear()


@pytest.mark.parametrize("kwargs", [dict(variant=1, in_type=1, out_dtype=0),   # one-CTA kernels: no FP8
                                    dict(variant=1, out_dtype=2),                 # nor int8 output
                                    dict(variant=3),                              # 3 names no kernel
                                    dict(variant=8), dict(variant=-1),
                                    dict(variant=2, out_dtype=2, beta_nonzero=True)])  # int8 output has no beta
def test_autotune_set_refuses_unbuilt(tc, kwargs):
    with pytest.raises(tc.TcgemmError):
        tc.binding.autotune_set(256, 256, 256, **kwargs)


def test_autotune_load_rejects_bad_files(tc, tmp_path):
    b = tc.binding
    b.autotune_clear()
    bad_header = tmp_path / "a.txt"
    bad_header.write_text("something else\n0 64 64 64 0 0 1 0 0 0 2\n")
    bad_line = tmp_path / "b.txt"
    bad_line.write_text("tcgemm-autotune 1\n0 64 64 64 0 0 1 0 0 0 2\n0 64 64 64 0 0 1 0 0 0 9\n")
    for p in (bad_header, bad_line, tmp_path / "missing.txt"):
        with pytest.raises(tc.TcgemmError):
            b.autotune_load(p)
    assert b.autotune_lookup(64, 64, 64) == 0        # nothing from the half-valid file was added
