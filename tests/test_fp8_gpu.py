"""GPU checks of the FP8 (e4m3) forward (fa_fwd_fp8, through the C ABI):
against the float64 model of its arithmetic (oracle/fp8.py) closely, and
against the exact oracle within the tolerance e4m3 allows.

Tolerances.  e4m3 keeps 4 significant bits: each rounding of Q, K (after the
block scale), V and P moves a value by up to 2^-4 of itself, so against the
exact result the output carries errors of several percent (rel-L2 about 5e-2
for O, up to ~0.1 in lse on these N(0, 1)-shaped inputs with scale
1/sqrt(128)).  Those errors belong to the FP8 algorithm, not to the kernel, so
the bound against the exact result is relative to the model's own error: the
kernel may exceed the model's rel-L2 (and lse max-abs) against the exact
result by at most 10% plus 2e-3 (5e-3 for lse), with absolute caps of 0.1
(0.2 for lse).  Against the model, which makes the same roundings, only the
kernel's fp32 arithmetic (exp2, accumulation order) and the bf16 output
differ, except where such a difference moves a value across an e4m3 rounding
boundary: rel-L2 <= 1e-2 for O, max-abs <= 1e-2 for lse.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as f8
from tests.parity import errors

pytestmark = pytest.mark.gpu

TOL_EXACT_RELL2 = 0.1   # absolute caps against the exact result
TOL_EXACT_LSE = 0.2
TOL_MODEL_RELL2 = 1e-2  # against the model of the same arithmetic
TOL_MODEL_LSE = 1e-2


def no_worse_than_model(err_kernel, err_model, slack):
    return err_kernel <= 1.1 * err_model + slack


@pytest.fixture(scope="module")
def fa(cuda_device):
    import exact_io_aware_35_gb300 as fa
    fa.load_library()
    return fa


def inputs(B, N, Hq, Hkv, seed, s=1.0, outliers=0.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, N, Hq, 128, generator=g) * s
    k = torch.randn(B, N, Hkv, 128, generator=g) * s
    v = torch.randn(B, N, Hkv, 128, generator=g)
    if outliers:
        # a few channels far larger than the rest (what rotation is for)
        q[..., :4] *= outliers
        k[..., :4] *= outliers
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def run(fa, q, k, v, causal, scale, rotate):
    o = torch.full_like(q.cuda(), float("nan"))
    lse = torch.full((q.shape[0], q.shape[2], q.shape[1]), float("nan"), device="cuda")
    fa.fa_fwd_fp8(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, rotate=rotate,
                  o=o, lse=lse)
    assert fa.fa_get_device_error() == fa.FA_OK
    return o.cpu(), lse.cpu()


CASES = [  # (B, N, Hq, Hkv, causal, rotate)
    (1, 300, 4, 2, True, True),
    (1, 300, 4, 2, False, False),
    (2, 128, 2, 1, True, False),
    (1, 1000, 8, 2, True, True),
    (1, 77, 2, 2, False, True),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,causal,rotate", CASES)
def test_fp8_matches_model_and_oracle(fa, B, N, Hq, Hkv, causal, rotate):
    q, k, v = inputs(B, N, Hq, Hkv, seed=N + Hq)
    scale = 1 / math.sqrt(128)
    o, lse = run(fa, q, k, v, causal, scale, rotate)
    o_m, lse_m = f8.attn_fwd_fp8(q, k, v, causal, scale, rotate)
    o_x, lse_x = oracle.attn_fwd(q, k, v, causal, scale)
    _, rel_m = errors(o, o_m)
    _, rel_x = errors(o, o_x)
    _, rel_mx = errors(o_m, o_x)  # the algorithm's own error
    lse_g = lse.double().numpy()
    lse_err, lse_err_m = np.abs(lse_g - lse_x).max(), np.abs(lse_m - lse_x).max()
    assert rel_m <= TOL_MODEL_RELL2, f"rel-L2 vs the fp8 model {rel_m:.3e}"
    assert np.abs(lse_g - lse_m).max() <= TOL_MODEL_LSE
    assert no_worse_than_model(rel_x, rel_mx, 2e-3), (rel_x, rel_mx)
    assert rel_x <= TOL_EXACT_RELL2, f"rel-L2 vs exact {rel_x:.3e}"
    assert no_worse_than_model(lse_err, lse_err_m, 5e-3), (lse_err, lse_err_m)
    assert lse_err <= TOL_EXACT_LSE


def test_rotation_reduces_error_with_outlier_channels(fa):
    # incoherent processing spreads the outlier channels over the row, so the
    # block scales stop being set by them
    q, k, v = inputs(1, 512, 4, 2, seed=70, s=0.5, outliers=20.0)
    scale = 1 / math.sqrt(128)
    o_x, _ = oracle.attn_fwd(q, k, v, True, scale)
    _, rel_plain = errors(run(fa, q, k, v, True, scale, False)[0], o_x)
    _, rel_rot = errors(run(fa, q, k, v, True, scale, True)[0], o_x)
    assert rel_rot < rel_plain, (rel_rot, rel_plain)


def test_fp8_bench_shape_sampled(fa):
    # the FP8 bench shape (gqa8k: B4 Hq32 Hkv8 N8192 d128 causal), batch
    # element 0: exact oracle at sampled rows
    from fa_workloads import WORKLOADS, make_inputs
    w = WORKLOADS["gqa8k"].with_(B=1)
    x = make_inputs(w, with_dout=False)
    o, lse = run(fa, x["q"], x["k"], x["v"], True, w.scale, True)
    rng = np.random.default_rng(71)
    rows = np.stack([np.zeros(64, int), rng.integers(0, w.Hq, 64), rng.integers(0, w.N, 64)], 1)
    rows[0] = (0, 0, 0)
    rows[1] = (0, w.Hq - 1, w.N - 1)
    o_r, lse_r = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], rows, True, w.scale)
    got = np.stack([o[0, i, h].double().numpy() for _, h, i in rows])
    lse_got = np.array([lse[0, h, i].item() for _, h, i in rows])
    rel = np.linalg.norm(got - o_r) / np.linalg.norm(o_r)
    assert rel <= TOL_EXACT_RELL2, rel
    assert np.abs(lse_got - lse_r).max() <= TOL_EXACT_LSE
    # the gqa8k recipe draws 0.5 N(0, 1): the algorithm's error is smaller there
    assert rel <= 5e-2, rel


def test_quantise_then_attend_equals_one_call(fa):
    q, k, v = inputs(1, 400, 4, 2, seed=72)
    o1, l1 = run(fa, q, k, v, True, 0.09, True)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.empty(fa.fa_fwd_fp8_workspace_size(1, 4, 2, 400, 128), dtype=torch.uint8,
                     device="cuda")
    o2 = torch.full_like(qd, float("nan"))
    l2 = torch.full((1, 4, 400), float("nan"), device="cuda")
    fa.fa_fwd_fp8(qd, kd, vd, causal=True, scale=0.09, o=o2, lse=l2, workspace=ws,
                  stage=fa.FA_FP8_QUANTIZE_ONLY)
    assert torch.isnan(o2).all()  # nothing but the copies
    fa.fa_fwd_fp8(qd, kd, vd, causal=True, scale=0.09, o=o2, lse=l2, workspace=ws,
                  stage=fa.FA_FP8_ATTEND_ONLY)
    assert fa.fa_get_device_error() == fa.FA_OK
    assert torch.equal(o1, o2.cpu()) and torch.equal(l1, l2.cpu())
