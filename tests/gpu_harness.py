"""Runs one GEMM case through the C ABI on the GPU with guard bands around C,
and compares the result with the oracle.  Used by the -m gpu tests and by the
package smoke check."""
from __future__ import annotations

import numpy as np
import torch

import gemm_inputs as gi
from tests import parity

GUARD_BYTES = 4096
SENTINEL_F32 = 0x7FC0DEAD  # a NaN bit pattern no kernel produces
SENTINEL_BF16 = 0x7FDE


class GuardedC:
    """C (N, ldc) inside a larger buffer; the bytes before and after it and
    the padding rows i >= M are filled with a sentinel and must stay intact."""

    def __init__(self, case: gi.GemmCase, device="cuda"):
        self.case = case
        f32 = case.out_dtype == gi.OUT_F32
        self.dtype = torch.float32 if f32 else torch.bfloat16
        self.itype = torch.int32 if f32 else torch.int16
        sentinel = SENTINEL_F32 if f32 else SENTINEL_BF16
        esz = 4 if f32 else 2
        self.guard = GUARD_BYTES // esz
        n_el = case.N * case.ldc
        self.buf = torch.empty(n_el + 2 * self.guard, dtype=self.dtype, device=device)
        self.buf.view(self.itype).fill_(sentinel if f32 else np.int16(np.uint16(sentinel)).item())
        self.C = self.buf[self.guard:self.guard + n_el].view(case.N, case.ldc)
        if case.beta != 0.0:
            self.C.copy_(case.C_in.to(device))
        else:
            self.C[:, :case.M] = float("nan")  # must never be read when beta == 0
        self.before = self.buf.view(self.itype).clone()

    def check_guards(self):
        after = self.buf.view(self.itype)
        g, M = self.guard, self.case.M
        assert torch.equal(after[:g], self.before[:g]), "write before C"
        assert torch.equal(after[-g:], self.before[-g:]), "write after C"
        if self.case.ldc > M:
            a = self.buf[g:g + self.case.N * self.case.ldc].view(self.itype).view(self.case.N, self.case.ldc)
            b = self.before[g:g + self.case.N * self.case.ldc].view(self.case.N, self.case.ldc)
            assert torch.equal(a[:, M:], b[:, M:]), "write into ldc padding rows"

    def result_np(self) -> np.ndarray:
        out = self.C[:, :self.case.M].contiguous().cpu()
        if self.dtype == torch.bfloat16:
            return out.view(torch.int16).numpy().view(np.uint16)
        return out.numpy()


def run_case(case: gi.GemmCase, variant: int = 0, stream=None) -> GuardedC:
    import tensor_core_matmul_gb300 as tc
    A = case.A.cuda()
    B = case.B.cuda()
    g = GuardedC(case)
    tc.gemm_bf16(A, B, g.C, case.alpha, case.beta, M=case.M, N=case.N, K=case.K,
                 stream=stream, variant=variant)
    torch.cuda.synchronize()
    st, where = tc.check_device_status()
    assert st == 0, f"device status {st} (role {where})"
    g.check_guards()
    return g


def record_stats(what: str, stats: dict) -> None:
    """Append one comparison's statistics as a JSON line to the file named by
    TCGEMM_PARITY_STATS, if set (for the record of second-clause counts)."""
    import json
    import os
    path = os.environ.get("TCGEMM_PARITY_STATS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, **stats}) + "\n")


def cin_np(case):
    if case.C_in is None:
        return None
    if case.C_in.dtype == torch.bfloat16:
        return gi.as_u16(case.C_in)
    return case.C_in.numpy()


def compare_full(o, case: gi.GemmCase, got: np.ndarray, exact: bool = False, what: str = ""):
    D = o.gemm_f64(case.M, case.N, case.K, gi.as_u16(case.A), gi.as_u16(case.B), cin_np(case),
                   case.alpha, case.beta)
    return _compare(o, case, got, D, None, None, exact, what)


def compare_sampled(o, case: gi.GemmCase, got: np.ndarray, rows: np.ndarray, cols: np.ndarray,
                    exact: bool = False, what: str = ""):
    D = o.gemm_sampled_f64(case.M, case.N, case.K, gi.as_u16(case.A), gi.as_u16(case.B), rows, cols,
                           cin_np(case), case.alpha, case.beta)
    return _compare(o, case, got[cols, rows], D, rows, cols, exact, what)


def _compare(o, case, got, D, rows, cols, exact, what):
    if case.out_dtype == gi.OUT_F32:
        if exact:
            parity.check_exact(got, o.round_f32(D), what)
            return {"size": int(np.size(got)), "exact": True}
        return parity.check_f32(got, D, case.K, what)
    else:
        ref = o.round_bf16(D)
        if exact:
            parity.check_exact(got, ref, what)
            return {"size": int(np.size(got)), "exact": True}
        else:
            def fallback(flat):
                if rows is None:  # the whole of C, flat in (N, M) order
                    c, r = np.divmod(flat.astype(np.int64), case.M)
                else:
                    r, c = rows.reshape(-1)[flat], cols.reshape(-1)[flat]
                G = o.absdot_sampled_f64(case.M, case.N, case.K, gi.as_u16(case.A), gi.as_u16(case.B), r, c)
                # |alpha| scales the product's error; beta*C adds one exact-ish term.
                return D.reshape(-1)[flat], abs(case.alpha) * G, case.K
            return parity.check_bf16(got, ref, what, fallback=fallback)
