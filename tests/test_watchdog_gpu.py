"""Bounded waits: a wait that nothing ever satisfies runs out, the kernel
records FA_ERR_DEVICE_TIMEOUT and returns, and the GPU stays usable.  Once one
wait of a launch has run out, every other pending wait of that launch gives up
at once, so a launch of many waves costs about one time limit, not one per
wave; and a failure left by an earlier launch does not stop a later one."""
import math
import time

import pytest
import torch

import fa_workloads as W

pytestmark = pytest.mark.gpu


def _forward(fa):
    w = W.Workload("t", 1, 2, 1, 256, 64, True, 1 / math.sqrt(64), seed=1)
    x = W.make_inputs(w, with_dout=False)
    return fa.fa_fwd(*(x[n].cuda() for n in ("q", "k", "v")), causal=True)


def _forward_is_clean(fa):
    o, lse = _forward(fa)
    assert fa.fa_get_device_error() == fa.FA_OK
    assert torch.isfinite(o.float()).all()
    return o, lse


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
    _forward_is_clean(fa)


def test_one_timeout_ends_a_multi_wave_launch(cuda_device):
    import exact_io_aware_35_gb300 as fa
    assert fa.fa_get_device_error() == fa.FA_OK
    limit_ns = 100_000_000  # 100 ms
    # far more blocks than the GPU holds at once (32 resident blocks of one
    # warp per SM at most): at least 8 waves, i.e. >= 0.8 s if each wave
    # waited out its own limit
    blocks = 8 * 32 * torch.cuda.get_device_properties(0).multi_processor_count + 1
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    fa.fa_debug_watchdog_probe(limit_ns, blocks)
    end.record()
    # a forward launched after the failed launch, before anyone read the
    # status, runs in full: the failure belongs to the probe's launch alone
    o, lse = _forward(fa)
    assert fa.fa_get_device_error() == fa.FA_ERR_DEVICE_TIMEOUT
    ms = start.elapsed_time(end)
    assert ms < 4 * limit_ns / 1e6, f"{blocks} blocks took {ms:.0f} ms for a {limit_ns / 1e6:.0f} ms limit"
    o_ref, lse_ref = _forward_is_clean(fa)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
