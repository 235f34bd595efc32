"""fa_bwd_noalloc -- the backward pass for callers that cannot allocate device
memory (a plug-in inside an application that owns all device allocations, or
a loop that must not call cudaMalloc mid-step) -- checked against fa_bwd with
a caller-owned workspace, on two calls in a row.

Both calls go through the C ABI.  The built-in scratch keeps the previous
call's contents, so the second call uses a different shape and inputs to show
nothing stale leaks into it.  This file sorts last so that a run stopping at
the first failure has already run every other test.
"""
import ctypes
import math

import pytest
import torch

import fa_workloads as W
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


def _noalloc(lib, t, B, H, Hkv, N, d, causal, scale):
    return lib.fa_bwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                              t["o"].data_ptr(), t["dout"].data_ptr(), t["lse"].data_ptr(),
                              t["dq"].data_ptr(), t["dk"].data_ptr(), t["dv"].data_ptr(),
                              t["o_lo"].data_ptr(), B, H, Hkv, N, d, int(causal),
                              ctypes.c_float(scale),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_fa_bwd_two_calls(cuda_device):
    import exact_io_aware_35_gb300 as fa
    lib = fa.load_library()
    cases = [(1, 4, 2, 700, 128, True, 41), (2, 6, 3, 513, 64, False, 42)]
    for B, H, Hkv, N, d, causal, seed in cases:
        w = W.Workload("t", B, H, Hkv, N, d, causal, 1.0 / math.sqrt(d), seed=seed)
        x = {n: t.cuda() for n, t in W.make_inputs(w).items()}
        o_lo = torch.empty_like(x["q"])
        o, lse = fa.fa_fwd(x["q"], x["k"], x["v"], causal=causal, o_lo=o_lo)
        ref = fa.fa_bwd(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=causal, o_lo=o_lo)
        t = dict(x, o=o, lse=lse, o_lo=o_lo, dq=torch.full_like(x["q"], float("nan")),
                 dk=torch.full_like(x["k"], float("nan")), dv=torch.full_like(x["v"], float("nan")))
        assert _noalloc(lib, t, B, H, Hkv, N, d, causal, w.scale) == fa.FA_OK
        assert fa.fa_get_device_error() == fa.FA_OK
        for name, got, want in zip(("dq", "dk", "dv"), (t["dq"], t["dk"], t["dv"]), ref):
            assert_close(got.cpu(), want.cpu(), name)


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
