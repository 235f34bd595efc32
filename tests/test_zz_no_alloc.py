"""fa_bwd_noalloc -- the backward pass for callers that cannot allocate device
memory (a plug-in inside an application that owns all device allocations, or
a loop that must not call cudaMalloc mid-step) -- checked through the C ABI
against the float64 oracle and against fa_bwd with a caller-owned workspace,
on two calls in a row.

The built-in scratch keeps the previous call's contents, so the second call
uses a different shape and inputs to show nothing stale leaks into it.

Accuracy.  fa_bwd_noalloc has no room for fp16 operand copies, so P and dS
enter their products rounded to bf16.  On N(0, 1) inputs that meets the
library's tolerances (max-abs 2e-2 beyond bf16 output rounding, rel-L2 5e-3).
On peaked rows (1% of the keys x8, where dS = P o (dP - D) nearly cancels and
|K| is large) the bf16 rounding of dS shows in dQ = dS K: there the entry
point meets rel-L2 5e-3 but not max-abs 2e-2, and the test holds it to the
documented limit NOALLOC_PEAKED_MAXABS instead.

This file sorts last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes
import math

import pytest
import torch

import fa_workloads as W
import oracle
from tests.parity import TOL_RELL2, assert_close, describe, error_report

pytestmark = pytest.mark.gpu

# max-abs error beyond bf16 output rounding of dQ, dK, dV on the peaked-row
# recipe (bf16 P and dS), the limit include/fa.h states for fa_bwd_noalloc
NOALLOC_PEAKED_MAXABS = 0.15


def _noalloc(lib, t, B, H, Hkv, N, d, causal, scale):
    return lib.fa_bwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                              t["o"].data_ptr(), t["dout"].data_ptr(), t["lse"].data_ptr(),
                              t["dq"].data_ptr(), t["dk"].data_ptr(), t["dv"].data_ptr(),
                              t["o_lo"].data_ptr(), B, H, Hkv, N, d, int(causal),
                              ctypes.c_float(scale),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _run(fa, lib, w):
    x_host = W.make_inputs(w)
    x = {n: t.cuda() for n, t in x_host.items()}
    o_lo = torch.empty_like(x["q"])
    o, lse = fa.fa_fwd(x["q"], x["k"], x["v"], causal=w.causal, scale=w.scale, o_lo=o_lo)
    t = dict(x, o=o, lse=lse, o_lo=o_lo, dq=torch.full_like(x["q"], float("nan")),
             dk=torch.full_like(x["k"], float("nan")), dv=torch.full_like(x["v"], float("nan")))
    assert _noalloc(lib, t, w.B, w.Hq, w.Hkv, w.N, w.d, w.causal, w.scale) == fa.FA_OK
    assert fa.fa_get_device_error() == fa.FA_OK
    return x_host, x, o, lse, o_lo, (t["dq"], t["dk"], t["dv"])


def test_noalloc_matches_oracle_and_fa_bwd_two_calls(cuda_device):
    import exact_io_aware_35_gb300 as fa
    lib = fa.load_library()
    cases = [(1, 4, 2, 700, 128, True, 41), (2, 6, 3, 513, 64, False, 42)]
    for B, H, Hkv, N, d, causal, seed in cases:
        w = W.Workload("t", B, H, Hkv, N, d, causal, 1.0 / math.sqrt(d), seed=seed)
        x_host, x, o, lse, o_lo, got = _run(fa, lib, w)
        exact = oracle.attn_bwd(x_host["q"], x_host["k"], x_host["v"], x_host["dout"], causal,
                                w.scale)
        ref = fa.fa_bwd(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=causal, o_lo=o_lo)
        for name, g, e, r in zip(("dq", "dk", "dv"), got, exact, ref):
            assert_close(g.cpu(), e, f"{name} vs oracle")
            assert_close(g.cpu(), r.cpu(), f"{name} vs fa_bwd")


def test_noalloc_peaked_rows_within_documented_limit(cuda_device):
    import exact_io_aware_35_gb300 as fa
    lib = fa.load_library()
    w = W.WORKLOADS["gqa32k_peaked"].with_(N=1024, Hq=8, Hkv=2)
    x_host, _, _, _, _, got = _run(fa, lib, w)
    exact = oracle.attn_bwd(x_host["q"], x_host["k"], x_host["v"], x_host["dout"], True, w.scale)
    for name, g, e in zip(("dq", "dk", "dv"), got, exact):
        maxabs, rell2, raw = error_report(g.cpu(), e)
        msg = describe(name, maxabs, rell2, raw) + f" (noalloc limit {NOALLOC_PEAKED_MAXABS})"
        print(msg)
        assert rell2 <= TOL_RELL2, msg
        assert maxabs <= NOALLOC_PEAKED_MAXABS, msg


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    import exact_io_aware_35_gb300 as fa
    lib = fa.load_library()
    x = torch.zeros(16, device="cuda")
    p = x.data_ptr()
    # B * H * N = 2^22 rows > the 2^21-row built-in scratch
    st = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, None, 1, 64, 64, 1 << 16, 128, 1,
                            ctypes.c_float(0.125), None)
    assert st == fa.FA_ERR_INVALID_ARG
    assert fa.fa_get_device_error() == fa.FA_OK
