"""GPU parity of fa_bwd (through the C ABI) against the float64 oracle.

The backward's inputs O and lse come from the forward; every expected value
comes from the oracle alone.
"""
import math

import numpy as np
import pytest
import torch

import fa_workloads as W
import oracle
from tests.guards import Guarded, check_all
from tests.parity import TOL_MAXABS, TOL_RELL2, assert_close, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import exact_io_aware_35_gb300 as fa
    fa.load_library()
    return fa


def run_bwd(fa, x, causal, scale, train=True):
    """Training pair: fa_fwd_train (o, o_lo, lse) then fa_bwd; train=False
    uses the plain forward and no o_lo.  Every buffer the library writes sits
    between guard canaries (tests/guards.py), checked after the launches."""
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    o = Guarded(q.shape, q.dtype, q.device)
    lse = Guarded((B, Hq, N), torch.float32, q.device)
    o_lo = Guarded(q.shape, q.dtype, q.device) if train else None
    wsb = fa.fa_bwd_workspace_size(B, Hq, Hkv, N, d)
    ws_f = Guarded((wsb,), torch.uint8, q.device, fill=255) if train else None
    fa.fa_fwd(q, k, v, causal=causal, scale=scale, o=o.t, lse=lse.t,
              o_lo=o_lo.t if train else None, workspace=ws_f.t if train else None)
    dq = Guarded(q.shape, q.dtype, q.device)
    dk = Guarded(k.shape, k.dtype, k.device)
    dv = Guarded(v.shape, v.dtype, v.device)
    ws = Guarded((wsb,), torch.uint8, q.device, fill=255)
    fa.fa_bwd(q, k, v, o.t, do, lse.t, causal=causal, scale=scale, dq=dq.t, dk=dk.t, dv=dv.t,
              workspace=ws.t, o_lo=o_lo.t if train else None)
    assert fa.fa_get_device_error() == fa.FA_OK
    check_all(o=o, lse=lse, o_lo=o_lo, fwd_workspace=ws_f, dq=dq, dk=dk, dv=dv, workspace=ws)
    return dq.t.cpu(), dk.t.cpu(), dv.t.cpu()


SHAPES = [
    (1, 1, 1, 128, 64, False),
    (1, 1, 1, 128, 128, True),
    (1, 2, 1, 1, 64, True),
    (1, 2, 2, 1, 128, False),
    (2, 4, 2, 300, 64, True),
    (2, 4, 2, 300, 64, False),
    (1, 4, 1, 257, 128, False),
    (1, 8, 2, 513, 128, True),
    (2, 3, 3, 700, 64, False),
    (1, 4, 4, 1024, 128, True),
    (1, 16, 1, 640, 128, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", SHAPES)
def test_bwd_matches_oracle(fa, B, Hq, Hkv, N, d, causal):
    w = W.Workload("t", B, Hq, Hkv, N, d, causal, 1.0 / math.sqrt(d), seed=200 + N + d)
    x = W.make_inputs(w)
    got = run_bwd(fa, x, causal, w.scale)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], causal, w.scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert_close(g, r, name)


def test_bwd_tiny_workload(fa):
    w = W.WORKLOADS["tiny"]
    x = W.make_inputs(w)
    got = run_bwd(fa, x, w.causal, w.scale)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], w.causal, w.scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert_close(g, r, name)


@pytest.fixture(scope="module")
def peaked_case(fa):
    # the peaked-row recipe (1% of K rows x8) at a size the oracle does in seconds
    w = W.WORKLOADS["gqa32k_peaked"].with_(N=1024, Hq=8, Hkv=2)
    x = W.make_inputs(w)
    got = run_bwd(fa, x, True, w.scale)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], True, w.scale)
    return got, ref


def test_bwd_peaked_rows_small_rel_l2(peaked_case):
    got, ref = peaked_case
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert errors(g, r)[1] <= TOL_RELL2, name


def test_bwd_peaked_rows_small_maxabs(peaked_case):
    # P and dS rounded to fp16 (3 more bits than bf16) before their products:
    # the x8 keys amplify the rounding of dS in dQ = dS K, of P^T in dV, of
    # dS^T in dK, and the training forward's P moves O and hence D
    got, ref = peaked_case
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert errors(g, r)[0] <= TOL_MAXABS, name


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_without_o_lo(fa, causal):
    # the plain forward's bf16 O alone is enough on unpeaked inputs
    w = W.Workload("t", 2, 4, 2, 384, 128, causal, 1 / math.sqrt(128), seed=31)
    x = W.make_inputs(w)
    got = run_bwd(fa, x, causal, w.scale, train=False)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], causal, w.scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert_close(g, r, name)


def test_fwd_train_matches_fwd(fa):
    # the training forward writes the same lse as the inference forward; its o
    # (P in fp16 for P V) is at least as close to the oracle, and o + o_lo is
    # its fp32 output to ~16 bits, closer still
    w = W.Workload("t", 1, 4, 2, 300, 128, True, 1 / math.sqrt(128), seed=32)
    x = W.make_inputs(w, with_dout=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = fa.fa_fwd(q, k, v, causal=True)
    o_lo = torch.empty_like(q)
    o2, l2 = fa.fa_fwd(q, k, v, causal=True, o_lo=o_lo)
    assert torch.equal(l1, l2)
    o_ref, _ = oracle.attn_fwd(x["q"], x["k"], x["v"], True, w.scale)
    inf_o = o1.cpu().double().numpy()
    hi = o2.cpu().double().numpy()
    lo = o_lo.cpu().double().numpy()
    assert_close(o2.cpu(), o_ref, "o (training forward)")
    assert np.linalg.norm(hi - o_ref) <= np.linalg.norm(inf_o - o_ref)
    assert np.abs(lo).max() <= np.abs(hi).max() * 2 ** -8
    # o_lo is O's rounding residual: it moves o toward the fp32 result, which
    # is closer to the exact output than the rounded o
    assert np.linalg.norm(hi + lo - o_ref) < 0.8 * np.linalg.norm(hi - o_ref)


def test_bwd_stages_match_single_call(fa):
    w = W.Workload("t", 1, 4, 2, 500, 128, True, 1 / math.sqrt(128), seed=33)
    x = W.make_inputs(w)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o_lo = torch.empty_like(q)
    o, lse = fa.fa_fwd(q, k, v, causal=True, o_lo=o_lo)
    a = fa.fa_bwd(q, k, v, o, do, lse, causal=True, o_lo=o_lo)
    ws = torch.empty(fa.fa_bwd_workspace_size(1, 4, 2, 500, 128), dtype=torch.uint8,
                     device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    # one stage per call, in the documented order (DQ writes the fp16 copy of
    # dout that DKDV reads)
    for st in (fa.FA_BWD_PREP, fa.FA_BWD_DSUM, fa.FA_BWD_DQ, fa.FA_BWD_DKDV):
        fa.fa_bwd(q, k, v, o, do, lse, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws,
                  stages=st, o_lo=o_lo)
    assert fa.fa_get_device_error() == fa.FA_OK
    for u, v_ in zip(a, (dq, dk, dv)):
        assert torch.equal(u, v_)


def test_bwd_after_fwd_train_reuses_copies(fa):
    # fa_fwd_train leaves the fp16 copies of q, k, v in the training workspace;
    # a backward on it that copies only dout gives exactly the standalone result
    w = W.Workload("t", 2, 4, 2, 333, 128, True, 1 / math.sqrt(128), seed=34)
    x = W.make_inputs(w)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    ws = torch.empty(fa.fa_bwd_workspace_size(2, 4, 2, 333, 128), dtype=torch.uint8,
                     device=q.device)
    o_lo = torch.empty_like(q)
    o, lse = fa.fa_fwd(q, k, v, causal=True, o_lo=o_lo, workspace=ws)
    a = fa.fa_bwd(q, k, v, o, do, lse, causal=True, o_lo=o_lo, workspace=ws,
                  stages=fa.FA_BWD_AFTER_FWD_TRAIN)
    b = fa.fa_bwd(q, k, v, o, do, lse, causal=True, o_lo=o_lo)
    # the same backward split as a timed training step splits it: max |dout|
    # with D, then dQ (with the copy of dout), then dK, dV
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for st in (fa.FA_BWD_PREP_DOUT | fa.FA_BWD_DSUM, fa.FA_BWD_DQ, fa.FA_BWD_DKDV):
        fa.fa_bwd(q, k, v, o, do, lse, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws,
                  stages=st, o_lo=o_lo)
    assert fa.fa_get_device_error() == fa.FA_OK
    for u, v_, w_ in zip(a, b, (dq, dk, dv)):
        assert torch.equal(u, v_)
        assert torch.equal(u, w_)


def test_bwd_deterministic(fa):
    w = W.Workload("t", 1, 8, 2, 700, 128, True, 1 / math.sqrt(128), seed=9)
    x = W.make_inputs(w)
    a = run_bwd(fa, x, True, w.scale)
    b = run_bwd(fa, x, True, w.scale)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
