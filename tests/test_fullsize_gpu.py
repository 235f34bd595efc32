"""Parity at the workloads' full sizes, in exactly the launch configuration
bench.py times, on outputs the oracle can compute one row at a time.

The bench-timed step (run_bench_step below mirrors bench.run_gpu): for the
workloads with a backward pass, the training forward (fa_fwd_train, P in
fp16, o_lo) on the training workspace, then the backward as three
fa_bwd_stage calls on that same workspace -- max |dO| with D
(FA_BWD_PREP_DOUT | FA_BWD_DSUM), dQ, then dK/dV -- run twice, as the bench's
warm-up and timed steps run back to back, with the outputs NaN-filled again
before the second step so that every element checked was written by it.
The forward-only workload (N=131072 MQA) times the inference fa_fwd.

Forward: sampled query rows (O row and lse) of every workload -- 256 rows for
the N=131072 MQA workload.  Backward: sampled dQ rows, and sampled dK / dV rows
of one (batch, kv head) group, whose exact values need that group's full row
statistics (the oracle computes them).  Row 0 and row N-1 are always in the
sample.  Every buffer the library writes sits between guard canaries
(tests/guards.py).  Each assertion message carries the raw max-abs error
beside the error beyond bf16 output rounding.
"""
import numpy as np
import pytest
import torch

import fa_workloads as W
import oracle
from tests.guards import Guarded, check_all
from tests.parity import TOL_LSE, TOL_MAXABS, TOL_RELL2, describe, error_report

pytestmark = pytest.mark.gpu

FWD_ROWS = {"tiny": 64, "gpt2s": 96, "gqa8k": 96, "gqa32k_peaked": 96, "mqa128k": 256}


@pytest.fixture(scope="module")
def fa(cuda_device):
    import exact_io_aware_35_gb300 as fa
    fa.load_library()
    return fa


def sample_rows(w: W.Workload, n: int, heads: int, seed: int):
    rng = np.random.default_rng(seed)
    rows = [(0, 0, 0), (w.B - 1, heads - 1, w.N - 1)]
    while len(rows) < n:
        rows.append((int(rng.integers(w.B)), int(rng.integers(heads)), int(rng.integers(w.N))))
    return np.array(rows, dtype=np.int64)


def run_bench_step(fa, w: W.Workload, steps: int = 2):
    """The bench's step on the workload's inputs, `steps` times in a row on
    the same buffers.  Returns (host inputs, o, lse, (dq, dk, dv) or None,
    the guarded buffers)."""
    x = W.make_inputs(w, with_dout=w.backward)
    dev = {n: t.cuda() for n, t in x.items()}
    q, k, v = dev["q"], dev["k"], dev["v"]
    g = {"o": Guarded(q.shape, q.dtype, q.device),
         "lse": Guarded((w.B, w.Hq, w.N), torch.float32, q.device)}
    if w.backward:
        g.update(o_lo=Guarded(q.shape, q.dtype, q.device),
                 dq=Guarded(q.shape, q.dtype, q.device),
                 dk=Guarded(k.shape, k.dtype, k.device),
                 dv=Guarded(v.shape, v.dtype, v.device),
                 workspace=Guarded((fa.fa_bwd_workspace_size(w.B, w.Hq, w.Hkv, w.N, w.d),),
                                   torch.uint8, q.device, fill=255))
    t = {n: b.t for n, b in g.items()}
    stages = (fa.FA_BWD_PREP_DOUT | fa.FA_BWD_DSUM, fa.FA_BWD_DQ, fa.FA_BWD_DKDV)
    for _ in range(steps):
        for n in ("o", "lse", "dq", "dk", "dv"):
            if n in t:
                t[n].fill_(float("nan"))
        if w.backward:
            fa.fa_fwd(q, k, v, causal=w.causal, scale=w.scale, o=t["o"], lse=t["lse"],
                      o_lo=t["o_lo"], workspace=t["workspace"])
            for st in stages:
                fa.fa_bwd(q, k, v, t["o"], dev["dout"], t["lse"], causal=w.causal,
                          scale=w.scale, dq=t["dq"], dk=t["dk"], dv=t["dv"],
                          workspace=t["workspace"], stages=st, o_lo=t["o_lo"])
        else:
            fa.fa_fwd(q, k, v, causal=w.causal, scale=w.scale, o=t["o"], lse=t["lse"])
    assert fa.fa_get_device_error() == fa.FA_OK
    check_all(**g)
    grads = (t["dq"], t["dk"], t["dv"]) if w.backward else None
    return x, dev, t["o"], t["lse"], grads, g


def check_rows(name, got, ref):
    maxabs, rell2, raw = error_report(got, ref)
    msg = describe(name, maxabs, rell2, raw)
    print(msg)
    assert maxabs <= TOL_MAXABS and rell2 <= TOL_RELL2, msg


def check_fwd_rows(w, x, o, lse, label):
    rows = sample_rows(w, FWD_ROWS[w.name], w.Hq, seed=7)
    b, h, i = (torch.from_numpy(rows[:, c]).cuda() for c in range(3))
    got_o = o[b, i, h].cpu()
    got_l = lse[b, h, i].cpu().double().numpy()
    ref_o, ref_l = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], rows, w.causal, w.scale)
    check_rows(f"{w.name} {label} o", got_o, ref_o)
    err = float(np.abs(got_l - ref_l).max())
    print(f"{w.name} {label} lse: max-abs {err:.3e} (tol {TOL_LSE})")
    assert err <= TOL_LSE, f"{w.name} {label} lse max-abs {err:.3e}"


@pytest.fixture(scope="module", params=W.WORKLOAD_ORDER)
def bench_run(fa, request):
    """One bench-path run per workload, shared by the forward and backward
    checks; pytest groups the tests by this module-scoped parameter, so each
    workload's buffers are released before the next workload runs."""
    w = W.WORKLOADS[request.param]
    torch.cuda.empty_cache()
    yield (w,) + run_bench_step(fa, w)
    torch.cuda.empty_cache()


def test_bench_forward_full_size_sampled_rows(bench_run):
    # the forward the bench times: fa_fwd_train for the training workloads
    # (d = 64 and 128, GQA, peaked rows), fa_fwd for the forward-only one
    w, x, _, o, lse, _, _ = bench_run
    check_fwd_rows(w, x, o, lse, "training forward" if w.backward else "forward")


def test_bench_backward_full_size_sampled_rows(bench_run):
    # the staged backward on the training forward's workspace, as timed
    w, x, _, _, _, grads, _ = bench_run
    if not w.backward:
        pytest.skip("forward-only workload")
    dq, dk, dv = grads
    qrows = sample_rows(w, 64, w.Hq, seed=11)
    # key rows of one (batch, kv head) group; its query heads' statistics are
    # computed in full by the oracle
    rng = np.random.default_rng(13)
    kvrows = np.array([(0, 0, 0), (0, 0, w.N - 1)] +
                      [(0, 0, int(j)) for j in rng.integers(w.N, size=30)], dtype=np.int64)
    ref = oracle.attn_bwd_rows(x["q"], x["k"], x["v"], x["dout"], qrows, kvrows, w.causal,
                               w.scale)
    qb, qh, qi = (torch.from_numpy(qrows[:, c]).cuda() for c in range(3))
    kb, kh, kj = (torch.from_numpy(kvrows[:, c]).cuda() for c in range(3))
    got = (dq[qb, qi, qh].cpu(), dk[kb, kj, kh].cpu(), dv[kb, kj, kh].cpu())
    for n, a, r in zip(("dq", "dk", "dv"), got, ref):
        check_rows(f"{w.name} {n}", a, r)


def test_single_call_backward_equals_bench_stages(fa, bench_run):
    # fa_bwd in one call on a fresh workspace (the fp16 copies of q, k, v made
    # by its own prep) gives bit for bit what the bench's staged backward on
    # the training forward's workspace gave, at the bench's full size
    w, x, dev, o, lse, grads, g = bench_run
    if w.name != "gqa8k":
        pytest.skip("checked on the bench workload")
    one = fa.fa_bwd(dev["q"], dev["k"], dev["v"], o, dev["dout"], lse, causal=w.causal,
                    scale=w.scale, o_lo=g["o_lo"].t)
    assert fa.fa_get_device_error() == fa.FA_OK
    for n, a, b in zip(("dq", "dk", "dv"), one, grads):
        assert torch.equal(a, b), n
    del one


@pytest.mark.parametrize("name", ["tiny", "gpt2s", "gqa8k", "gqa32k_peaked"])
def test_inference_forward_full_size_sampled_rows(fa, name):
    # fa_fwd (bf16 P, no o_lo, no workspace) at the same sizes
    w = W.WORKLOADS[name]
    x = W.make_inputs(w, with_dout=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = Guarded(q.shape, q.dtype, q.device)
    lse = Guarded((w.B, w.Hq, w.N), torch.float32, q.device)
    fa.fa_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o.t, lse=lse.t)
    assert fa.fa_get_device_error() == fa.FA_OK
    check_all(o=o, lse=lse)
    check_fwd_rows(w, x, o.t, lse.t, "inference forward")
