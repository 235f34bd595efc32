"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, not against the oracle's own formula.

Each test is chosen so that a plausible mistake in the oracle (dropped term,
wrong sign or index, transposed operand, wrong mask side, missing GQA sum)
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import fa_workloads as W
import oracle
from oracle import numpy_oracle as npo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, s=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * s


def qkv(B=2, N=13, Hq=4, Hkv=2, d=8, seed=0, s=1.0):
    return rnd((B, N, Hq, d), seed, s), rnd((B, N, Hkv, d), seed + 1, s), rnd((B, N, Hkv, d), seed + 2, s)


@pytest.mark.parametrize("causal", [False, True])
def test_c_oracle_matches_numpy_oracle(causal):
    q, k, v = qkv(B=2, N=37, Hq=4, Hkv=2, d=8, seed=3)
    do = rnd(q.shape, 9)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.3)
    o2, lse2 = npo.attn_fwd(q, k, v, causal, 0.3)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)
    g = oracle.attn_bwd(q, k, v, do, causal, 0.3)
    g2 = npo.attn_bwd(q, k, v, do, causal, 0.3)
    for a, b in zip(g, g2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    # With V = [I_N | 0] the output's first N columns are P itself.
    N, d = 9, 16
    q = rnd((1, N, 1, d), 1)
    k = rnd((1, N, 1, d), 2)
    v = np.zeros((1, N, 1, d))
    v[0, :, 0, :N] = np.eye(N)
    o, _ = oracle.attn_fwd(q, k, v, causal, 0.7)
    P = o[0, :, 0, :N]
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (P >= 0).all()
    np.testing.assert_allclose(o[0, :, 0, N:], 0.0, atol=0)
    if causal:
        assert np.all(P[np.triu_indices(N, 1)] == 0.0)
        assert np.all(P[np.tril_indices(N)] > 0.0)
    np.testing.assert_allclose(P, npo.attn_probs(q, k, causal, 0.7), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal):
    q, k, _ = qkv(seed=4)
    c = rnd((1, 1, 2, 8), 5)
    v = np.broadcast_to(c, (2, 13, 2, 8)).copy()
    o, _ = oracle.attn_fwd(q, k, v, causal, 0.5)
    for h in range(4):
        np.testing.assert_allclose(o[:, :, h, :], np.broadcast_to(c[0, 0, h // 2], (2, 13, 8)),
                                   rtol=0, atol=1e-12)


def test_single_key_gives_o_equal_v():
    q, k, v = qkv(N=1, seed=6)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.25)
        for h in range(4):
            np.testing.assert_allclose(o[:, 0, h], v[:, 0, h // 2], rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[:, h, 0],
                                       0.25 * np.einsum("bc,bc->b", q[:, 0, h], k[:, 0, h // 2]),
                                       rtol=0, atol=1e-13)


def test_causal_first_row_is_first_value():
    q, k, v = qkv(N=17, seed=7)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.5)
    for h in range(4):
        np.testing.assert_allclose(o[:, 0, h], v[:, 0, h // 2], rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_mean_of_visible_values(causal):
    N = 11
    q, k, v = qkv(N=N, seed=8)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.0)
    for h in range(4):
        vh = v[:, :, h // 2]
        if causal:
            expect = np.cumsum(vh, axis=1) / np.arange(1, N + 1)[None, :, None]
            lexp = np.log(np.arange(1, N + 1))[None, :]
        else:
            expect = np.broadcast_to(vh.mean(axis=1, keepdims=True), vh.shape)
            lexp = np.full((1, N), math.log(N))
        np.testing.assert_allclose(o[:, :, h], expect, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, h], np.broadcast_to(lexp, (2, N)), rtol=0, atol=1e-13)


@pytest.mark.parametrize("a,b", [(0.3, -1.7), (4.0, 2.5), (-6.0, 0.0)])
def test_closed_form_two_keys(a, b):
    # Q = [[a],[b]], K = [[1],[0]], V = [[1],[0]], scale 1: scores [q_i, 0],
    # so O_i = sigmoid(q_i) and lse_i = ln(1 + e^{q_i}) without the mask;
    # with it, row 0 sees key 0 only: O_0 = 1, lse_0 = a.
    q = np.array([a, b]).reshape(1, 2, 1, 1)
    k = np.array([1.0, 0.0]).reshape(1, 2, 1, 1)
    v = np.array([1.0, 0.0]).reshape(1, 2, 1, 1)
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))
    sp = lambda x: math.log1p(math.exp(x))
    o, lse = oracle.attn_fwd(q, k, v, False, 1.0)
    np.testing.assert_allclose(o.ravel(), [sig(a), sig(b)], rtol=1e-13)
    np.testing.assert_allclose(lse.ravel(), [sp(a), sp(b)], rtol=1e-13)
    o, lse = oracle.attn_fwd(q, k, v, True, 1.0)
    np.testing.assert_allclose(o.ravel(), [1.0, sig(b)], rtol=1e-13)
    np.testing.assert_allclose(lse.ravel(), [a, sp(b)], rtol=1e-13)


def test_joint_key_value_permutation_invariance():
    q, k, v = qkv(N=19, seed=10)
    perm = np.random.default_rng(11).permutation(19)
    o, lse = oracle.attn_fwd(q, k, v, False, 0.4)
    o2, lse2 = oracle.attn_fwd(q, k[:, perm], v[:, perm], False, 0.4)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_common_key_offset_shifts_only_lse(causal):
    # Adding one vector u to every key row adds scale*q_i.u to a whole row of
    # scores: softmax is unchanged, lse_i moves by exactly that amount.
    q, k, v = qkv(N=15, seed=12)
    u = rnd((1, 1, 2, 8), 13)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.6)
    o2, lse2 = oracle.attn_fwd(q, k + u, v, causal, 0.6)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    shift = np.stack([0.6 * np.einsum("bnc,c->bn", q[:, :, h], u[0, 0, h // 2]) for h in range(4)],
                     axis=1)
    np.testing.assert_allclose(lse2 - lse, shift, rtol=0, atol=1e-12)


def test_two_block_merge_equals_full():
    # The two-block update of the online softmax ("FlashAttention 1, 2, and 3
    # Explained", section 2): l_new = e^{m1-m} l1 + e^{m2-m} l2 and
    # O_new = diag(e^{m1-m}) O1 + (block-2 contribution), then normalised.
    # Written here with lse = m + ln l of each half.
    q, k, v = qkv(N=24, seed=14)
    o, lse = oracle.attn_fwd(q, k, v, False, 0.5)
    # query rows 0..11 against keys 0..11 and keys 12..23 separately
    o1, l1 = oracle.attn_fwd(q[:, :12], k[:, :12], v[:, :12], False, 0.5)
    o2, l2 = oracle.attn_fwd(q[:, :12], k[:, 12:], v[:, 12:], False, 0.5)
    m = np.maximum(l1, l2)
    a1, a2 = np.exp(l1 - m), np.exp(l2 - m)
    lsum = a1 + a2
    a1t = np.transpose(a1, (0, 2, 1))[..., None]
    a2t = np.transpose(a2, (0, 2, 1))[..., None]
    om = (a1t * o1 + a2t * o2) / np.transpose(lsum, (0, 2, 1))[..., None]
    np.testing.assert_allclose(om, o[:, :12], rtol=0, atol=1e-13)
    np.testing.assert_allclose(m + np.log(lsum), lse[:, :, :12], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_with_repeated_kv(causal):
    B, N, Hq, Hkv, d = 2, 11, 6, 2, 5
    q, k, v = qkv(B, N, Hq, Hkv, d, seed=15)
    do = rnd(q.shape, 16)
    g = Hq // Hkv
    kr, vr = np.repeat(k, g, axis=2), np.repeat(v, g, axis=2)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.45)
    o2, lse2 = oracle.attn_fwd(q, kr, vr, causal, 0.45)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-14)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.45)
    dq2, dk2, dv2 = oracle.attn_bwd(q, kr, vr, do, causal, 0.45)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, N, Hkv, g, d).sum(3), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(B, N, Hkv, g, d).sum(3), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_differences(causal):
    B, N, Hq, Hkv, d = 1, 6, 2, 1, 3
    q, k, v = qkv(B, N, Hq, Hkv, d, seed=17)
    do = rnd(q.shape, 18)
    scale = 0.8
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, scale)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, causal, scale)
        return float((o * do).sum())

    h = 1e-6
    base = {"q": q, "k": k, "v": v}
    for name, g in (("q", dq), ("k", dk), ("v", dv)):
        x = base[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            plus, minus = dict(base), dict(base)
            plus[name], minus[name] = x.copy(), x.copy()
            plus[name][idx] += h
            minus[name][idx] -= h
            fd[idx] = (loss(plus["q"], plus["k"], plus["v"])
                       - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        err = np.abs(fd - g).max() / max(np.abs(g).max(), 1e-30)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_identities(causal):
    B, N, Hq, Hkv, d = 2, 14, 4, 2, 6
    q, k, v = qkv(B, N, Hq, Hkv, d, seed=19)
    do = rnd(q.shape, 20)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.5)
    # each row of dS sums to zero  =>  sum over keys of dK vanishes
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    # rows of P sum to one  =>  sum over keys of dV = sum over queries of dO (per group)
    np.testing.assert_allclose(dv.sum(axis=1), do.reshape(B, N, Hkv, 2, d).sum(axis=(1, 3)),
                               rtol=0, atol=1e-12)
    # all keys equal  =>  dQ = scale * k * rowsum(dS) = 0
    kc = np.broadcast_to(k[:, :1], k.shape).copy()
    dq0, _, _ = oracle.attn_bwd(q, kc, v, do, causal, 0.5)
    np.testing.assert_allclose(dq0, 0.0, atol=1e-13)


def test_row_sampled_entry_points_match_full():
    B, N, Hq, Hkv, d = 2, 21, 4, 2, 8
    q, k, v = qkv(B, N, Hq, Hkv, d, seed=21)
    do = rnd(q.shape, 22)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.5)
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.5)
        rows = np.array([[0, 0, 0], [1, 3, 20], [0, 2, 7], [1, 1, 13]])
        orow, lrow = oracle.attn_fwd_rows(q, k, v, rows, causal, 0.5)
        for r, (b, h, i) in enumerate(rows):
            np.testing.assert_array_equal(orow[r], o[b, i, h])
            assert lrow[r] == lse[b, h, i]
        kvrows = np.array([[0, 0, 0], [1, 1, 20], [1, 0, 9]])
        dqr, dkr, dvr = oracle.attn_bwd_rows(q, k, v, do, rows, kvrows, causal, 0.5)
        for r, (b, h, i) in enumerate(rows):
            np.testing.assert_allclose(dqr[r], dq[b, i, h], rtol=0, atol=1e-14)
        for r, (b, h, j) in enumerate(kvrows):
            np.testing.assert_allclose(dkr[r], dk[b, j, h], rtol=0, atol=1e-14)
            np.testing.assert_allclose(dvr[r], dv[b, j, h], rtol=0, atol=1e-14)


def test_bf16_inputs_are_taken_exactly():
    import torch
    w = W.WORKLOADS["tiny"].with_(N=5)
    x = W.make_inputs(w)
    o, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], w.causal, w.scale)
    o2, lse2 = npo.attn_fwd(x["q"].to(torch.float64).numpy(), x["k"].to(torch.float64).numpy(),
                            x["v"].to(torch.float64).numpy(), w.causal, w.scale)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)


def test_memory_wall_arithmetic_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "memory_wall_n16384.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, val = line.split()
                vals[key] = float(val)
    N = int(vals["N"])
    assert W.score_matrix_elements(N) == int(vals["elements"])
    assert W.score_matrix_bytes(N, 2) == int(vals["bytes_per_head_2byte"])
    assert math.floor(W.score_matrix_bytes(N, 2) / 1e5) / 10 == vals["page_megabytes"]


# ---- Nq queries against Nk keys (the split-KV decode entry) ----

@pytest.mark.parametrize("causal", [False, True])
def test_kv_oracle_with_equal_lengths_is_the_square_oracle(causal):
    q, k, v = qkv(N=17, seed=30)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.4)
    o2, lse2 = oracle.attn_fwd_kv(q, k, v, causal, 0.4)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_kv_oracle_matches_numpy(causal):
    q = rnd((2, 5, 6, 8), 31)
    k, v = rnd((2, 23, 2, 8), 32), rnd((2, 23, 2, 8), 33)
    o, lse = oracle.attn_fwd_kv(q, k, v, causal, 0.3)
    o2, lse2 = npo.attn_fwd_kv(q, k, v, causal, 0.3)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def test_kv_causal_queries_are_the_last_rows_of_the_square_problem():
    # the reading of the causal mask for Nq < Nk: the Nq queries are the last
    # Nq positions of the sequence, so they equal the last rows of the square
    # causal problem over all Nk positions
    Nk, Nq = 29, 6
    qf, k, v = qkv(N=Nk, seed=34)
    o, lse = oracle.attn_fwd(qf, k, v, True, 0.45)
    o2, lse2 = oracle.attn_fwd_kv(qf[:, Nk - Nq:], k, v, True, 0.45)
    np.testing.assert_allclose(o2, o[:, Nk - Nq:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse[:, :, Nk - Nq:], rtol=0, atol=1e-13)


def test_kv_single_causal_query_sees_every_key():
    q = rnd((1, 1, 4, 8), 35)
    k, v = rnd((1, 40, 2, 8), 36), rnd((1, 40, 2, 8), 37)
    oc, lc = oracle.attn_fwd_kv(q, k, v, True, 0.5)
    on, ln = oracle.attn_fwd_kv(q, k, v, False, 0.5)
    np.testing.assert_array_equal(oc, on)
    np.testing.assert_array_equal(lc, ln)


def _merge_in_order(parts):
    # the online-softmax update applied chunk after chunk, each chunk given as
    # its normalised output and lse ("FlashAttention 1, 2, and 3 Explained",
    # section 2, the two-block l and O update): running (m, l, unnormalised O)
    m = l = acc = None
    for o_c, lse_c in parts:
        lse_t = np.transpose(lse_c, (0, 2, 1))[..., None]  # [B, Nq, Hq, 1]
        if m is None:
            m, l, acc = lse_t, np.ones_like(lse_t), o_c.copy()
            continue
        m_new = np.maximum(m, lse_t)
        a_old, a_new = np.exp(m - m_new), np.exp(lse_t - m_new)
        acc = (a_old * l * acc + a_new * o_c) / (a_old * l + a_new)
        l = a_old * l + a_new
        m = m_new
    return acc, np.transpose((m + np.log(l))[..., 0], (0, 2, 1))


@pytest.mark.parametrize("causal", [False, True])
def test_chunked_kv_merge_in_order_equals_full(causal):
    # ring attention's per-chunk results, merged in ring order, equal the
    # whole; chunks may be empty for a causal query (lse = -inf there)
    Nq, Nk = 4, 37
    q = rnd((2, Nq, 4, 8), 38)
    k, v = rnd((2, Nk, 2, 8), 39), rnd((2, Nk, 2, 8), 40)
    o, lse = oracle.attn_fwd_kv(q, k, v, causal, 0.35)
    bounds = [0, 10, 11, 25, Nk]
    parts = []
    for c0, c1 in zip(bounds[:-1], bounds[1:]):
        # keys [c0, c1): the queries keep their positions Nk - Nq + i, so a
        # causal chunk sees keys j <= Nk - Nq + i, i.e. the square problem's
        # mask shifted by the chunk start
        kc, vc = k[:, c0:c1], v[:, c0:c1]
        if causal:
            # chunk key j' = c0 + j is visible iff c0 + j <= Nk - Nq + i
            oc, lc = npo.attn_fwd_kv(q, kc, vc, False, 0.35)
            vis = (np.arange(c0, c1)[None, :] <= (Nk - Nq) + np.arange(Nq)[:, None])
            oc = np.zeros_like(oc)
            lc = np.full_like(lc, -np.inf)
            for b in range(2):
                for h in range(4):
                    s = 0.35 * (q[b, :, h] @ kc[b, :, h // 2].T)
                    s = np.where(vis, s, -np.inf)
                    for i in range(Nq):
                        if not vis[i].any():
                            continue
                        mm = s[i].max()
                        e = np.exp(s[i] - mm)
                        lc[b, h, i] = mm + np.log(e.sum())
                        oc[b, i, h] = (e / e.sum()) @ vc[b, :, h // 2]
        else:
            oc, lc = oracle.attn_fwd_kv(q, kc, vc, False, 0.35)
        parts.append((oc, lc))
    om, lm = _merge_in_order(parts)
    np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)


# ---- block-sparse forward (a block mask over bs x bs blocks) ----

def _mask(Hq, nb, seed, density=0.5):
    return (np.random.default_rng(seed).random((Hq, nb, nb)) < density).astype(np.uint8)


@pytest.mark.parametrize("causal", [False, True])
def test_blockmask_all_ones_is_dense(causal):
    q, k, v = qkv(N=23, seed=50)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.4)
    m = np.ones((4, 6, 6), dtype=np.uint8)  # blocks of 4, nb = 6
    o2, lse2 = oracle.attn_fwd_blockmask(q, k, v, m, 4, causal, 0.4)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_blockmask_c_matches_numpy(causal):
    q, k, v = qkv(N=30, seed=51)
    m = _mask(4, 4, seed=52)  # blocks of 8 over N = 30 (ragged last block)
    o, lse = oracle.attn_fwd_blockmask(q, k, v, m, 8, causal, 0.3)
    o2, lse2 = npo.attn_fwd_blockmask(q, k, v, m, 8, causal, 0.3)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(lse2))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lse[fin], lse2[fin], rtol=0, atol=1e-12)


def test_blockmask_block_diagonal_is_independent_blocks():
    # each query block sees only its own key block: attention block by block
    q, k, v = qkv(N=24, seed=53)
    m = np.zeros((4, 3, 3), dtype=np.uint8)
    for i in range(3):
        m[:, i, i] = 1
    o, lse = oracle.attn_fwd_blockmask(q, k, v, m, 8, False, 0.5)
    for i in range(3):
        sl = slice(8 * i, 8 * i + 8)
        ob, lb = oracle.attn_fwd(q[:, sl], k[:, sl], v[:, sl], False, 0.5)
        np.testing.assert_allclose(o[:, sl], ob, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, sl], lb, rtol=0, atol=1e-13)


def test_blockmask_empty_rows_are_zero_and_minus_infinity():
    q, k, v = qkv(N=16, seed=54)
    m = np.ones((4, 2, 2), dtype=np.uint8)
    m[1, 1, :] = 0       # head 1, query block 1: nothing visible
    m[2, 0, 0] = 0       # head 2, query block 0 under causal: only block 0 is visible -> empty
    o, lse = oracle.attn_fwd_blockmask(q, k, v, m, 8, True, 0.5)
    assert (o[:, 8:, 1] == 0).all() and np.isneginf(lse[:, 1, 8:]).all()
    assert (o[:, :8, 2] == 0).all() and np.isneginf(lse[:, 2, :8]).all()
    assert np.isfinite(lse[:, 0]).all() and np.isfinite(lse[:, 3]).all()


def test_blockmask_rows_merge_from_their_blocks():
    # a query row under a block mask is the in-order merge of its visible
    # blocks' separate results: the split-KV merge applied to a sparse row
    q, k, v = qkv(N=32, seed=55)
    m = _mask(4, 4, seed=56, density=0.6)
    m[:, :, 0] = 1  # every row sees at least block 0
    o, lse = oracle.attn_fwd_blockmask(q, k, v, m, 8, False, 0.45)
    for h in range(4):
        for qb in range(4):
            parts = []
            for kb in range(4):
                if not m[h, qb, kb]:
                    continue
                sl = slice(8 * kb, 8 * kb + 8)
                oc, lc = oracle.attn_fwd_kv(q[:, 8 * qb:8 * qb + 8], k[:, sl], v[:, sl], False, 0.45)
                parts.append((oc, lc))
            om, lm = _merge_in_order(parts)
            np.testing.assert_allclose(om[:, :, h], o[:, 8 * qb:8 * qb + 8, h], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lm[:, h], lse[:, h, 8 * qb:8 * qb + 8], rtol=0, atol=1e-12)


# ---- the FP8 model (block quantisation, incoherent processing) ----

from oracle import fp8 as f8  # noqa: E402


def test_e4m3_rounding_fixes_every_value_and_ties_go_even():
    vals = f8.e4m3_values()
    assert len(vals) == 254 and vals.max() == 448.0 and vals[vals > 0].min() == 2.0 ** -9
    np.testing.assert_array_equal(f8.e4m3_round(vals), vals)
    pos = np.unique(vals[vals >= 0])
    mids = (pos[:-1] + pos[1:]) / 2
    got = f8.e4m3_round(mids)
    # a midpoint goes to the neighbour whose mantissa is even
    lo_even = np.array([int(round(p / 2.0 ** (max(np.floor(np.log2(p)), -6) - 3))) % 2 == 0
                        if p > 0 else True for p in pos[:-1]])
    np.testing.assert_array_equal(got, np.where(lo_even, pos[:-1], pos[1:]))
    # nearest otherwise, and saturation
    x = np.random.default_rng(60).uniform(-500, 500, 2000)
    y = f8.e4m3_round(x)
    inside = np.abs(x) <= 448
    nearest = vals[np.abs(x[inside, None] - vals[None, :]).argmin(axis=1)]
    np.testing.assert_array_equal(np.abs(y[inside]), np.abs(nearest))
    assert (np.abs(y[~inside]) == 448).all()


def test_hadamard_rotation_preserves_scores():
    H = f8.hadamard()
    np.testing.assert_array_equal(H @ H.T, 128 * np.eye(128))
    s = f8.rot_signs()
    assert set(np.unique(s)) == {-1.0, 1.0}
    q, k = rnd((7, 128), 61), rnd((9, 128), 62)
    qr, kr = (q * s) @ H.T, (k * s) @ H.T
    np.testing.assert_allclose(qr @ kr.T, 128 * (q @ k.T), rtol=1e-12, atol=1e-10)


@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_model_without_rounding_is_exact_attention(rotate, causal):
    # with the e4m3 rounding switched off, the model's rotation, block scales,
    # lazy-rescaled online softmax and normalisation give the exact result
    q, k, v = rnd((1, 300, 4, 128), 63), rnd((1, 300, 2, 128), 64), rnd((1, 300, 2, 128), 65)
    o, lse = f8.attn_fwd_fp8(q, k, v, causal, 0.09, rotate, quantize=False)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 0.09)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-11)


def test_fp8_block_scales_map_block_maxima_to_448():
    x = rnd((1, 200, 2, 128), 66) * np.array([1.0, 50.0])[None, None, :, None]
    y = f8.quantize_blocks(x, rotate=False)
    for h in range(2):
        for r0 in (0, 128):
            blk, yb = x[0, r0:r0 + 128, h], y[0, r0:r0 + 128, h]
            i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            # the maximum maps to 448, which e4m3 holds exactly
            assert abs(yb[i] - blk[i]) <= 1e-12 * abs(blk[i])
            assert np.abs(yb - blk).max() <= np.abs(blk).max() * 2.0 ** -4
