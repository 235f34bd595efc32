"""GPU parity of fa_fwd (through the C ABI) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import fa_workloads as W
import oracle
from tests.guards import Guarded, check_all
from tests.parity import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import exact_io_aware_35_gb300 as fa
    fa.load_library()
    return fa


def run_fwd(fa, x, causal, scale):
    """fa_fwd with NaN-filled outputs between guard canaries (tests/guards.py)."""
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    B, N, Hq, d = q.shape
    o = Guarded(q.shape, q.dtype, q.device)
    lse = Guarded((B, Hq, N), torch.float32, q.device)
    fa.fa_fwd(q, k, v, causal=causal, scale=scale, o=o.t, lse=lse.t)
    assert fa.fa_get_device_error() == fa.FA_OK
    check_all(o=o, lse=lse)
    return o.t.cpu(), lse.t.cpu()


# (B, Hq, Hkv, N, d, causal): several tiles, ragged tails, N=1, GQA and MQA
SHAPES = [
    (1, 1, 1, 128, 64, False),
    (1, 1, 1, 128, 128, False),
    (1, 2, 2, 1, 64, True),
    (1, 2, 1, 1, 128, False),
    (2, 4, 2, 300, 64, True),
    (2, 4, 2, 300, 64, False),
    (1, 4, 1, 257, 128, False),
    (1, 8, 2, 513, 128, True),
    (2, 3, 3, 700, 64, False),
    (1, 4, 4, 1024, 128, True),
    (1, 16, 1, 640, 128, True),
    # more (batch, head, 256-row block) items than the GB300 has SMs (152):
    # every persistent CTA takes two to four items, longest first when causal
    (2, 48, 8, 600, 128, True),
    (1, 80, 10, 530, 128, False),
    (2, 64, 8, 520, 64, True),
    (1, 96, 96, 400, 64, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", SHAPES)
def test_fwd_matches_oracle(fa, B, Hq, Hkv, N, d, causal):
    w = W.Workload("t", B, Hq, Hkv, N, d, causal, 1.0 / math.sqrt(d), seed=100 + N + d)
    x = W.make_inputs(w, with_dout=False)
    o, lse = run_fwd(fa, x, causal, w.scale)
    o_ref, lse_ref = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, w.scale)
    assert_close(o, o_ref, "o")
    assert_lse_close(lse, lse_ref)


def test_fwd_tiny_workload(fa):
    w = W.WORKLOADS["tiny"]
    x = W.make_inputs(w, with_dout=False)
    o, lse = run_fwd(fa, x, w.causal, w.scale)
    o_ref, lse_ref = oracle.attn_fwd(x["q"], x["k"], x["v"], w.causal, w.scale)
    assert_close(o, o_ref, "o")
    assert_lse_close(lse, lse_ref)


def test_fwd_peaked_rows_small(fa):
    # peaked-row recipe (1% of K rows x8) at a size the oracle does in seconds:
    # stresses the lazy rescale of the running max
    w = W.WORKLOADS["gqa32k_peaked"].with_(N=1536, Hq=8, Hkv=2)
    x = W.make_inputs(w, with_dout=False)
    o, lse = run_fwd(fa, x, True, w.scale)
    o_ref, lse_ref = oracle.attn_fwd(x["q"], x["k"], x["v"], True, w.scale)
    assert_close(o, o_ref, "o")
    assert_lse_close(lse, lse_ref)


def test_fwd_deterministic(fa):
    w = W.Workload("t", 1, 4, 2, 777, 128, True, 1 / math.sqrt(128), seed=7)
    x = W.make_inputs(w, with_dout=False)
    a = run_fwd(fa, x, True, w.scale)
    b = run_fwd(fa, x, True, w.scale)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
