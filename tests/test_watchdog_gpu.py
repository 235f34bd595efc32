"""Bounded waits: a wait that nothing ever satisfies runs out, the kernel
records FA_ERR_DEVICE_TIMEOUT and returns, and the GPU stays usable."""
import math
import time

import pytest
import torch

import fa_workloads as W

pytestmark = pytest.mark.gpu


def test_watchdog_times_out_and_gpu_recovers(cuda_device):
    import exact_io_aware_35_gb300 as fa
    assert fa.fa_get_device_error() == fa.FA_OK
    t0 = time.time()
    fa.fa_debug_watchdog_probe(50_000_000)  # 50 ms limit
    st = fa.fa_get_device_error()
    assert st == fa.FA_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 5.0
    assert fa.fa_get_device_error() == fa.FA_OK  # reading cleared it
    # the context is intact: a normal forward still runs and is clean
    w = W.Workload("t", 1, 2, 1, 256, 64, True, 1 / math.sqrt(64), seed=1)
    x = W.make_inputs(w, with_dout=False)
    o, lse = fa.fa_fwd(*(x[n].cuda() for n in ("q", "k", "v")), causal=True)
    assert fa.fa_get_device_error() == fa.FA_OK
    assert torch.isfinite(o.float()).all()
