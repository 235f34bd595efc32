"""Parity at the workloads' full sizes, in the launch configuration bench.py
times, on outputs the oracle can compute one row at a time.

Forward: sampled query rows (O row and lse) of every workload -- 256 rows for
the N=131072 MQA workload.  Backward: sampled dQ rows, and sampled dK / dV rows
of one (batch, kv head) group, whose exact values need that group's full row
statistics (the oracle computes them).  Row 0 and row N-1 are always in the
sample.
"""
import numpy as np
import pytest
import torch

import fa_workloads as W
import oracle
from tests.parity import TOL_LSE, TOL_MAXABS, TOL_RELL2, errors

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


def run(fa, w: W.Workload, backward: bool):
    x = W.make_inputs(w, with_dout=backward)
    dev = {n: t.cuda() for n, t in x.items()}
    o_lo = torch.empty_like(dev["q"]) if backward else None
    o, lse = fa.fa_fwd(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale, o_lo=o_lo)
    grads = None
    if backward:
        grads = fa.fa_bwd(dev["q"], dev["k"], dev["v"], o, dev["dout"], lse, causal=w.causal,
                          scale=w.scale, o_lo=o_lo)
    assert fa.fa_get_device_error() == fa.FA_OK
    return x, o, lse, grads


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_forward_full_size_sampled_rows(fa, name):
    w = W.WORKLOADS[name]
    x, o, lse, _ = run(fa, w, backward=False)
    rows = sample_rows(w, FWD_ROWS[name], w.Hq, seed=7)
    b, h, i = (torch.from_numpy(rows[:, c]) for c in range(3))
    got_o = o[b.cuda(), i.cuda(), h.cuda()].cpu()
    got_l = lse[b.cuda(), h.cuda(), i.cuda()].cpu()
    ref_o, ref_l = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], rows, w.causal, w.scale)
    maxabs, rell2 = errors(got_o, ref_o)
    assert maxabs <= TOL_MAXABS and rell2 <= TOL_RELL2, (maxabs, rell2)
    assert np.abs(got_l.double().numpy() - ref_l).max() <= TOL_LSE


def _bwd_samples(fa, name):
    w = W.WORKLOADS[name]
    x, o, lse, (dq, dk, dv) = run(fa, w, backward=True)
    qrows = sample_rows(w, 64, w.Hq, seed=11)
    g = w.Hq // w.Hkv
    # key rows of one (batch, kv head) group; its query heads' statistics are
    # computed in full by the oracle
    rng = np.random.default_rng(13)
    kvrows = np.array([(0, 0, 0), (0, 0, w.N - 1)] +
                      [(0, 0, int(j)) for j in rng.integers(w.N, size=30)], dtype=np.int64)
    ref_dq, ref_dk, ref_dv = oracle.attn_bwd_rows(x["q"], x["k"], x["v"], x["dout"], qrows,
                                                  kvrows, w.causal, w.scale)
    qb, qh, qi = (torch.from_numpy(qrows[:, c]).cuda() for c in range(3))
    kb, kh, kj = (torch.from_numpy(kvrows[:, c]).cuda() for c in range(3))
    got = (dq[qb, qi, qh].cpu(), dk[kb, kj, kh].cpu(), dv[kb, kj, kh].cpu())
    return got, (ref_dq, ref_dk, ref_dv)


@pytest.mark.parametrize("name", ["tiny", "gpt2s", "gqa8k"])
def test_backward_full_size_sampled_rows(fa, name):
    got, ref = _bwd_samples(fa, name)
    for n, a, r in zip(("dq", "dk", "dv"), got, ref):
        maxabs, rell2 = errors(a, r)
        assert maxabs <= TOL_MAXABS and rell2 <= TOL_RELL2, (n, maxabs, rell2)


@pytest.fixture(scope="module")
def peaked_bwd(fa):
    return _bwd_samples(fa, "gqa32k_peaked")


def test_backward_peaked_full_size_rel_l2(peaked_bwd):
    got, ref = peaked_bwd
    for n, a, r in zip(("dq", "dk", "dv"), got, ref):
        assert errors(a, r)[1] <= TOL_RELL2, n


def test_backward_peaked_full_size_maxabs(peaked_bwd):
    # P and dS enter their products in fp16 (training forward and fa_bwd)
    got, ref = peaked_bwd
    for n, a, r in zip(("dq", "dk", "dv"), got, ref):
        assert errors(a, r)[0] <= TOL_MAXABS, n
