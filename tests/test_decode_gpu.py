"""GPU parity of the split-KV forward (fa_fwd_splitkv, through the C ABI)
against the float64 oracle's Nq-queries-against-Nk-keys forward."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.guards import Guarded, check_all
from tests.parity import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import exact_io_aware_35_gb300 as fa
    fa.load_library()
    return fa


def inputs(B, Nq, Nk, Hq, Hkv, d, seed, s=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, Nq, Hq, d, generator=g) * s).to(torch.bfloat16)
    k = (torch.randn(B, Nk, Hkv, d, generator=g) * s).to(torch.bfloat16)
    v = torch.randn(B, Nk, Hkv, d, generator=g).to(torch.bfloat16)
    return q, k, v


def run(fa, q, k, v, causal, scale, splits):
    """fa_fwd_splitkv with NaN-filled outputs and its fp32 workspace between
    guard canaries (tests/guards.py)."""
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    o = Guarded(qd.shape, qd.dtype, qd.device)
    lse = Guarded((B, Hq, Nq), torch.float32, qd.device)
    wsb = fa.fa_fwd_splitkv_workspace_size(B, Hq, Hkv, Nq, Nk, d, causal, splits)
    ws = Guarded((wsb,), torch.uint8, qd.device, fill=255) if wsb else None
    fa.fa_fwd_splitkv(qd, kd, vd, causal=causal, scale=scale, num_splits=splits, o=o.t,
                      lse=lse.t, workspace=ws.t if ws else None)
    assert fa.fa_get_device_error() == fa.FA_OK
    check_all(o=o, lse=lse, workspace=ws)
    return o.t.cpu(), lse.t.cpu()


# (B, Nq, Nk, Hq, Hkv, d, causal, splits): decode (Nq = 1), a few queries, several
# query tiles (Nq above 128 / g), ragged and short key lengths, MHA, GQA, MQA,
# one split (direct write), several, and the library's choice
CASES = [
    (2, 1, 1000, 8, 2, 128, True, 0),
    (2, 1, 1000, 8, 2, 128, False, 3),
    (2, 1, 1000, 8, 2, 128, True, 1),
    (1, 1, 50, 4, 4, 128, True, 0),
    (1, 5, 777, 8, 2, 64, True, 4),
    (1, 200, 3000, 2, 2, 64, True, 0),
    (2, 40, 257, 16, 2, 128, True, 2),
    (1, 3, 4096, 32, 1, 128, False, 0),
    (1, 130, 130, 1, 1, 128, True, 2),
    (3, 7, 2049, 6, 3, 64, False, 0),
]


@pytest.mark.parametrize("B,Nq,Nk,Hq,Hkv,d,causal,splits", CASES)
def test_splitkv_matches_oracle(fa, B, Nq, Nk, Hq, Hkv, d, causal, splits):
    q, k, v = inputs(B, Nq, Nk, Hq, Hkv, d, seed=B * 1000 + Nq * 7 + Nk, s=0.5)
    scale = 1 / math.sqrt(d)
    o, lse = run(fa, q, k, v, causal, scale, splits)
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, causal, scale)
    assert_close(o, o_ref, "o")
    assert_lse_close(lse, lse_ref)


def test_split_counts_agree(fa):
    # every split count gives the oracle's result; the merge is exact up to
    # fp32 rounding, so the counts also agree with each other closely
    q, k, v = inputs(2, 1, 2000, 8, 2, 128, seed=5)
    outs = [run(fa, q, k, v, True, 0.1, s) for s in (1, 2, 5, 16)]
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, True, 0.1)
    for o, lse in outs:
        assert_close(o, o_ref, "o")
        assert_lse_close(lse, lse_ref)
    base = outs[0][0].float()
    for o, _ in outs[1:]:
        assert (o.float() - base).abs().max().item() <= 2 ** -7


def test_square_problem_matches_fa_fwd(fa):
    # Nq == Nk: the split-KV forward computes fa_fwd's result
    q, k, v = inputs(1, 300, 300, 4, 2, 128, seed=6)
    o1, l1 = run(fa, q, k, v, True, 0.09, 0)
    o2, l2 = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=0.09)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 0.09)
    assert_close(o1, o_ref, "splitkv o")
    assert_close(o2.cpu(), o_ref, "fa_fwd o")
    assert np.abs(l1.numpy() - l2.cpu().numpy()).max() <= 2e-3


def test_peaked_keys(fa):
    # 1% of keys x8: the rescale path (the reference max moves within a split)
    # and splits whose maxima differ by far more than fp32's range of e^x
    q, k, v = inputs(1, 2, 5000, 8, 2, 128, seed=7)
    idx = torch.randperm(5000, generator=torch.Generator().manual_seed(8))[:50]
    k = k.float()
    k[:, idx] *= 8
    k = k.to(torch.bfloat16)
    o, lse = run(fa, q, k, v, True, 1 / math.sqrt(128), 0)
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, True, 1 / math.sqrt(128))
    assert_close(o, o_ref, "o")
    assert_lse_close(lse, lse_ref)


def test_decode_bench_shape_sampled(fa):
    # the decode bench shape (B8 Hq32 Hkv8, Nq 1, Nk 32768, d 128, causal):
    # whole-output oracle on two batch elements
    B, Nq, Nk, Hq, Hkv, d = 8, 1, 32768, 32, 8, 128
    q, k, v = inputs(B, Nq, Nk, Hq, Hkv, d, seed=9)
    o, lse = run(fa, q, k, v, True, 1 / math.sqrt(d), 0)
    for b in (0, B - 1):
        o_ref, lse_ref = oracle.attn_fwd_kv(q[b:b + 1], k[b:b + 1], v[b:b + 1], True,
                                            1 / math.sqrt(d))
        assert_close(o[b:b + 1], o_ref, f"o[b={b}]")
        assert_lse_close(lse[b:b + 1], lse_ref)


def test_ring_chunks_merged_in_order(fa):
    # The math ring attention depends on, on one GPU with no communication:
    # each key/value chunk's (O_c, lse_c) from its own call, merged on the host
    # in ring order with the two-block online-softmax update, equals the whole.
    # Queries are the sequence's last Nq positions (causal): every chunk before
    # the last is fully visible, the last one carries the causal edge.
    B, Nq, Nk, Hq, Hkv, d = 2, 3, 1500, 8, 2, 128
    q, k, v = inputs(B, Nq, Nk, Hq, Hkv, d, seed=11)
    scale = 1 / math.sqrt(d)
    bounds = [0, 256, 600, 1100, Nk]
    m = l = acc = None
    for c0, c1 in zip(bounds[:-1], bounds[1:]):
        last = c1 == Nk
        o_c, lse_c = run(fa, q, k[:, c0:c1].contiguous(), v[:, c0:c1].contiguous(), last, scale, 1)
        o_c = o_c.double().numpy()
        lse_t = np.transpose(lse_c.double().numpy(), (0, 2, 1))[..., None]
        if m is None:
            m, l, acc = lse_t, np.ones_like(lse_t), o_c
            continue
        m_new = np.maximum(m, lse_t)
        a_old, a_new = np.exp(m - m_new), np.exp(lse_t - m_new)
        acc = (a_old * l * acc + a_new * o_c) / (a_old * l + a_new)
        l = a_old * l + a_new
        m = m_new
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, True, scale)
    assert_close(acc, o_ref, "merged o")
    assert_lse_close(np.transpose((m + np.log(l))[..., 0], (0, 2, 1)), lse_ref)
