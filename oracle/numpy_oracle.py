"""Independent float64 numpy oracle for exact attention.

TEST INFRASTRUCTURE ONLY (imported by tests/, the smoke check and bench.py's
cpu_baseline leg).  It shares no code with the C oracle in attn_oracle.c and
none with the CUDA library; it exists so that the two CPU oracles can be
cross-checked against each other.

Forward: the definition O = softmax(scale * Q K^T [+ causal mask]) V
("FlashAttention and the Kernel Era", section "The Mathematics", first
equation; "FlashAttention 1, 2, and 3 Explained", section 1, the S/P/O
equations), written with whole-matrix numpy operations per (batch, head):
materialise S, subtract the row max, exponentiate, normalise, multiply by V.

Backward: the derivative of that definition for L = sum(O * dO)
(dV = P^T dO, dP = dO V^T, D = rowsum(P o dP), dS = P o (dP - D),
dQ = scale dS K, dK = scale dS^T Q; GQA groups summed).  The pages print no
gradient formulas; this is the calculus of the forward definition.

Layout: q, dout [B, N, Hq, d]; k, v [B, N, Hkv, d]; lse [B, Hq, N].
"""
from __future__ import annotations

import numpy as np


def _head_scores(qh: np.ndarray, kh: np.ndarray, causal: bool, scale: float) -> np.ndarray:
    s = scale * (qh @ kh.T)
    if causal:
        n = s.shape[0]
        s = np.where(np.tril(np.ones((n, n), dtype=bool)), s, -np.inf)
    return s


def _softmax_rows(s: np.ndarray):
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return e / l, (m + np.log(l))[:, 0]


def attn_fwd(q, k, v, causal: bool, scale: float):
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            s = _head_scores(q[b, :, h], k[b, :, h // g], causal, scale)
            p, lse[b, h] = _softmax_rows(s)
            o[b, :, h] = p @ v[b, :, h // g]
    return o, lse


def attn_fwd_kv(q, k, v, causal: bool, scale: float):
    """Nq queries against Nk keys; causal: query i sees keys j <= i + Nk - Nq."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    vis = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            s = scale * (q[b, :, h] @ k[b, :, h // g].T)
            if causal:
                s = np.where(vis, s, -np.inf)
            p, lse[b, h] = _softmax_rows(s)
            o[b, :, h] = p @ v[b, :, h // g]
    return o, lse


def attn_fwd_blockmask(q, k, v, block_mask, block: int, causal: bool, scale: float):
    """Block-sparse forward: element mask = block mask expanded (and causal);
    empty rows give O = 0, lse = -inf."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    blk = np.arange(N) // block
    o = np.zeros_like(q)
    lse = np.full((B, Hq, N), -np.inf)
    for h in range(Hq):
        vis = np.asarray(block_mask[h])[blk[:, None], blk[None, :]] != 0
        if causal:
            vis &= np.tril(np.ones((N, N), dtype=bool))
        rows = vis.any(axis=1)
        for b in range(B):
            s = np.where(vis, scale * (q[b, :, h] @ k[b, :, h // g].T), -np.inf)
            s = s[rows]
            p, l = _softmax_rows(s)
            o[b, rows, h] = p @ v[b, :, h // g]
            lse[b, h, rows] = l
    return o, lse


def attn_probs(q, k, causal: bool, scale: float, b: int = 0, h: int = 0) -> np.ndarray:
    """The probability matrix P of one (batch, head), for invariant checks."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    g = q.shape[2] // k.shape[2]
    p, _ = _softmax_rows(_head_scores(q[b, :, h], k[b, :, h // g], causal, scale))
    return p


def attn_bwd(q, k, v, dout, causal: bool, scale: float):
    q, k, v, dout = (np.asarray(t, dtype=np.float64) for t in (q, k, v, dout))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, :, h // g], v[b, :, h // g]
            p, _ = _softmax_rows(_head_scores(q[b, :, h], kh, causal, scale))
            do = dout[b, :, h]
            dp = do @ vh.T
            D = (p * dp).sum(axis=1, keepdims=True)
            ds = p * (dp - D)
            dq[b, :, h] = scale * (ds @ kh)
            dk[b, :, h // g] += scale * (ds.T @ q[b, :, h])
            dv[b, :, h // g] += p.T @ do
    return dq, dk, dv
