"""Float64 model of the FP8 (e4m3) attention forward -- TEST INFRASTRUCTURE ONLY.

Imported by tests/ only; it shares no code with the CUDA library.  The FP8
forward is an approximation of attention, so besides the exact oracle the
tests compare it with this model of its arithmetic, written from the method's
description ("FlashAttention and the Kernel Era", the FP8 paragraph;
"FlashAttention 1, 2, and 3 Explained", section 4: FP8 with block
quantisation and incoherent processing), step by step in that order:

1. incoherent processing (optional): every row of Q and K is multiplied by
   diag(s) H, H the 128 x 128 Walsh-Hadamard matrix (Sylvester order,
   unnormalised: H H^T = 128 I) and s fixed signs, so Q K^T is unchanged up
   to the factor 128, which the softmax scale absorbs;
2. block quantisation: each 128-row block of each head of Q and K is scaled
   so that its largest magnitude maps to 448 (the largest e4m3) and rounded
   to e4m3; V gets one such scale per head;
3. the online softmax over 128-key blocks with the lazy rescale (the
   reference maximum moves only when a block's maximum exceeds it by more
   than 2^8), P = 2^(x - m_ref) rounded to e4m3 for the P V product while the
   row sum uses the unrounded P;
4. O = (sum_j P8_j V8_j) * sv / l and lse = (m_ref + log2 l) ln 2.

e4m3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; normal values 2^-6 ..
448, subnormals multiples of 2^-9; round to nearest, ties to even;
saturating at +-448 (the conversion the kernels use).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (bf16 -> float64 is exact)
        import torch
        x = x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # quantum: 2^(e - 3) in the binade [2^e, 2^(e+1)) for e >= -6, 2^-9 below
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    q = np.exp2(e - 3.0)
    y = np.round(a / q) * q  # numpy rounds half to even
    y = np.minimum(y, E4M3_MAX)
    return np.copysign(y, x)


def e4m3_values() -> np.ndarray:
    """The 254 finite values of e4m3 (both zeros), from the bit layout."""
    vals = []
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        if e == 15 and m == 7:
            continue  # NaN
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.append(-v if s else v)
    return np.array(vals)


def rot_signs(n: int = 128) -> np.ndarray:
    """s_c = -1 when the top bit of c * 2654435761 (mod 2^32) is set."""
    c = np.arange(n, dtype=np.uint64)
    top = ((c * np.uint64(2654435761)) & np.uint64(0xFFFFFFFF)) >> np.uint64(31)
    return np.where(top == 1, -1.0, 1.0)


def hadamard(n: int = 128) -> np.ndarray:
    """H[k, c] = (-1)^popcount(k & c)."""
    k = np.arange(n)[:, None] & np.arange(n)[None, :]
    pop = np.zeros_like(k)
    while k.any():
        pop += k & 1
        k >>= 1
    return np.where(pop % 2 == 1, -1.0, 1.0)


def quantize_blocks(x: np.ndarray, rotate: bool, quantize: bool = True):
    """x [B, N, H, 128] -> (values after rotation and e4m3 rounding, scaled
    back to their magnitude), one scale per 128-row block of each head."""
    x = _f64(x)
    if rotate:
        x = (x * rot_signs()) @ hadamard().T
    B, N, H, d = x.shape
    out = np.empty_like(x)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, 128):
                blk = x[b, r0:r0 + 128, h]
                m = float(np.abs(blk).max())
                s = m / E4M3_MAX if m > 0 else 1.0
                out[b, r0:r0 + 128, h] = (e4m3_round(blk / s) if quantize else blk / s) * s
    return out


def quantize_heads(v: np.ndarray, quantize: bool = True):
    """v [B, N, H, 128] with one scale per head."""
    v = _f64(v)
    out = np.empty_like(v)
    for b in range(v.shape[0]):
        for h in range(v.shape[2]):
            m = float(np.abs(v[b, :, h]).max())
            s = m / E4M3_MAX if m > 0 else 1.0
            out[b, :, h] = (e4m3_round(v[b, :, h] / s) if quantize else v[b, :, h] / s) * s
    return out


# The reference maximum of the online softmax moves only when a block's
# maximum exceeds it by more than this many log2 units (a factor 2^8).
LAZY_THRESHOLD = 8.0


def row_sum_terms(p: np.ndarray) -> np.ndarray:
    """What the running row sum l adds for one block: the unrounded P."""
    return p


def pv_operand(p: np.ndarray, quantize: bool) -> np.ndarray:
    """P as it enters the P V product: rounded to e4m3, no scale (P <= 2^8)."""
    return e4m3_round(p) if quantize else p


def attn_fwd_fp8(q, k, v, causal: bool, scale: float, rotate: bool, quantize: bool = True):
    """The model of fa_fwd_fp8.  Returns (o [B,N,Hq,d], lse [B,Hq,N])."""
    q8 = quantize_blocks(q, rotate, quantize)
    k8 = quantize_blocks(k, rotate, quantize)
    v8 = quantize_heads(v, quantize)
    sl2 = scale * np.log2(np.e) / (128.0 if rotate else 1.0)
    B, N, Hq, d = q8.shape
    g = Hq // k8.shape[2]
    o = np.zeros((B, N, Hq, d))
    lse = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            x_all = sl2 * (q8[b, :, h] @ k8[b, :, h // g].T)  # [N, N], log2 units
            for i in range(N):
                lim = i if causal else N - 1
                m_ref, l, acc = -np.inf, 0.0, np.zeros(d)
                for j0 in range(0, lim + 1, 128):
                    x = x_all[i, j0:min(j0 + 128, lim + 1)]
                    m_new = max(m_ref, float(x.max()))
                    if m_new > m_ref + LAZY_THRESHOLD:
                        alpha = np.exp2(m_ref - m_new) if np.isfinite(m_ref) else 0.0
                        l *= alpha
                        acc *= alpha
                        m_ref = m_new
                    p = np.exp2(x - m_ref)
                    l += row_sum_terms(p).sum()
                    acc += pv_operand(p, quantize) @ v8[b, j0:j0 + len(x), h // g]
                o[b, i, h] = acc / l
                lse[b, h, i] = (m_ref + np.log2(l)) * np.log(2.0)
    return o, lse
