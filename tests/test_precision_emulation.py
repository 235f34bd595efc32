"""Why P and dS enter their products in fp16: a float64 emulation of the
kernels' rounding steps on the peaked-row recipe, against the exact oracle.

The emulation follows the arithmetic of the training forward and backward
step by step, with every intermediate that the kernels round rounded the same
way and everything else exact: the forward's online softmax over 128-key
blocks with the lazy rescale (the reference maximum moves only when a block's
maximum exceeds it by more than 8 in log2 units), P = 2^(x - m_ref) rounded
for O += P V while the row sum takes the unrounded P, O rounded to bf16 and
its residual o_lo = bf16(O - o); then D = rowsum(dO (o + o_lo)), P recomputed
from lse, dP = dO V^T, dS = P (dP - D) rounded for dQ = scale dS K and
dK = scale dS^T Q, and P rounded for dV = P^T dO.  "Rounded" is bf16 for the
bf16 operand path (fa_fwd, fa_bwd_noalloc) and fp16 (behind the exact
power-of-two range scaling the library applies) for the fp16 path (fa_fwd_train
and fa_bwd).

On the peaked recipe (1% of the keys x8, N 1024, Hq 8, Hkv 2) the bf16 path
misses max-abs 2e-2 on dQ (0.279 beyond bf16 output rounding) -- dS =
P o (dP - D) nearly cancels on the peaked keys, and dQ = dS K multiplies its
rounding by |K| ~ 90 -- while the fp16 path meets it (0.017).  Both meet
rel-L2 5e-3.  The GPU tests check the
kernels themselves; this pins the design choice to arithmetic anyone can
rerun on a CPU.
"""
import numpy as np
import pytest

import fa_workloads as W
import oracle
from tests.parity import TOL_MAXABS, TOL_RELL2, errors


def round_bf16(x):
    """float64 -> nearest bf16 (ties to even, through float32), as float64."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def round_fp16_scaled(x, bound):
    """fp16 rounding behind a power-of-two scaling that puts `bound` just
    under 2^15, undone exactly (the library's operand copies)."""
    s = 2.0 ** (15 - np.ceil(np.log2(bound))) if bound > 0 else 1.0
    return np.asarray(x * s, dtype=np.float16).astype(np.float64) / s


def emulate(q, k, v, do, scale, op):
    """q, do [N, Hq, d], k, v [N, Hkv, d] (float64 holding bf16 values);
    causal.  op: 'bf16' or 'fp16'.  Returns (dq, dk, dv) in float64."""
    N, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    l2e = np.log2(np.e)
    vmax = np.abs(v).max()
    domax = np.abs(do).max()

    def rnd_p(p):  # P <= 2^8 under the lazy rescale
        return round_bf16(p) if op == "bf16" else round_fp16_scaled(p, 256.0)

    def rnd_ds(x):  # |dS| <= 2 d max|dO| max|V|
        return round_bf16(x) if op == "bf16" else round_fp16_scaled(x, 2 * d * domax * vmax)

    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    mask = np.tril(np.ones((N, N), dtype=bool))
    for h in range(Hq):
        hk = h // g
        x = scale * l2e * (q[:, h] @ k[:, hk].T)  # log2 units
        x = np.where(mask, x, -np.inf)
        # forward: online softmax over 128-key blocks, lazy rescale
        m_ref = np.full(N, -np.inf)
        l = np.zeros(N)
        acc = np.zeros((N, d))
        for j0 in range(0, N, 128):
            xb = x[:, j0:j0 + 128]
            m_new = np.maximum(m_ref, xb.max(axis=1))
            move = m_new > m_ref + 8.0
            alpha = np.where(move, np.exp2(np.where(np.isfinite(m_ref), m_ref - m_new, -np.inf)), 1.0)
            l *= alpha
            acc *= alpha[:, None]
            m_ref = np.where(move, m_new, m_ref)
            p = np.exp2(xb - m_ref[:, None])
            l += p.sum(axis=1)
            acc += rnd_p(p) @ v[j0:j0 + 128, hk]
        o32 = acc / l[:, None]
        o = round_bf16(o32)
        o_lo = round_bf16(o32 - o)
        lse2 = m_ref + np.log2(l)
        # backward
        D = ((o + o_lo) * do[:, h]).sum(axis=1)
        p = np.exp2(x - lse2[:, None])
        dp = do[:, h] @ v[:, hk].T
        ds = rnd_ds(p * (dp - D[:, None]))
        dq[:, h] = scale * (ds @ k[:, hk])
        dk[:, hk] += scale * (ds.T @ q[:, h])
        dv[:, hk] += rnd_p(p).T @ do[:, h]
    return dq, dk, dv


@pytest.fixture(scope="module")
def peaked():
    w = W.WORKLOADS["gqa32k_peaked"].with_(N=1024, Hq=8, Hkv=2)
    x = W.make_inputs(w)
    f = {n: t[0].double().numpy() for n, t in x.items()}
    exact = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], True, w.scale)
    return w, f, [e[0] for e in exact]


@pytest.mark.parametrize("op", ["bf16", "fp16"])
def test_emulated_operand_path_on_peaked_rows(peaked, op):
    w, f, exact = peaked
    got = emulate(f["q"], f["k"], f["v"], f["dout"], w.scale, op)
    res = {n: errors(g, e) for n, g, e in zip(("dq", "dk", "dv"), got, exact)}
    print(op, {n: f"max-abs {m:.3e} rel-L2 {r:.3e}" for n, (m, r) in res.items()})
    for n, (maxabs, rell2) in res.items():
        assert rell2 <= TOL_RELL2, (op, n, rell2)
    if op == "bf16":
        # the bf16 operands miss the max-abs bound on dQ
        assert res["dq"][0] > TOL_MAXABS, res["dq"]
    else:
        for n, (maxabs, _) in res.items():
            assert maxabs <= TOL_MAXABS, (n, maxabs)
