"""Seeded synthetic workloads for exact attention, plus work/byte accounting.

This module holds no attention arithmetic.  It is the one module that both
the CPU oracle's tests and the CUDA path's tests/bench import: it only draws
inputs and counts nominal FLOPs and bytes.

Inputs are drawn on the CPU with torch.Generator(seed), in the order Q, K, V,
dO, as float32 N(0, 1) samples, multiplied by the workload's value scale and
rounded to bf16 (round-to-nearest-even), so every machine sees the same bits.
Layout is [B, N, H, d] (the flash_attn_func layout on the "Flash Attention"
page, section "Code Example").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    scale: float
    value_scale: float = 1.0     # multiplies the N(0,1) draws of Q, K, V
    peaked_frac: float = 0.0     # fraction of K rows multiplied by peaked_mult
    peaked_mult: float = 1.0
    backward: bool = True
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _s(d: int) -> float:
    return 1.0 / math.sqrt(d)


# The five workloads: tiny; GPT-2-small-shaped (B16 H12 N2048 d64, the shape of
# the "Flash Attention" page's benchmark paragraph); causal GQA at N=8192;
# long-context causal GQA with peaked rows; very long causal MQA (forward only).
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 128, 64, False, _s(64), seed=0),
    "gpt2s": Workload("gpt2s", 16, 12, 12, 2048, 64, False, _s(64), seed=1),
    "gqa8k": Workload("gqa8k", 4, 32, 8, 8192, 128, True, _s(128), value_scale=0.5, seed=2),
    "gqa32k_peaked": Workload("gqa32k_peaked", 1, 32, 8, 32768, 128, True, _s(128),
                              peaked_frac=0.01, peaked_mult=8.0, seed=3),
    "mqa128k": Workload("mqa128k", 1, 16, 1, 131072, 128, True, _s(128), backward=False, seed=4),
}
WORKLOAD_ORDER = ["tiny", "gpt2s", "gqa8k", "gqa32k_peaked", "mqa128k"]


@dataclass(frozen=True)
class DecodeWorkload:
    """Nq queries (the last Nq positions of a sequence) against Nk keys and
    values: the split-KV decode shape."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    scale: float
    seed: int = 0

    def with_(self, **kw) -> "DecodeWorkload":
        return replace(self, **kw)


# Decode against a long cache: GQA at 32k (8 sequences, one new token each),
# MQA at 128k (the long-context workload's head layout).
DECODE_WORKLOADS = {
    "decode32k": DecodeWorkload("decode32k", 8, 32, 8, 1, 32768, 128, True, _s(128), seed=5),
    "decode128k_mqa": DecodeWorkload("decode128k_mqa", 1, 16, 1, 1, 131072, 128, True, _s(128),
                                     seed=6),
}


def describe_decode(w: DecodeWorkload) -> str:
    return (f"B{w.B} Hq{w.Hq} Hkv{w.Hkv} Nq{w.Nq} Nk{w.Nk} d{w.d} "
            f"{'causal' if w.causal else 'non-causal'} scale={w.scale:.6g}")


def make_decode_inputs(w: DecodeWorkload):
    """q [B, Nq, Hq, d], k, v [B, Nk, Hkv, d]: bf16 N(0, 1) draws in that order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = torch.randn((w.B, w.Nq, w.Hq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Nk, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Nk, w.Hkv, w.d), generator=g, dtype=torch.float32)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}


def decode_flops(w: DecodeWorkload) -> float:
    """4 * d FLOPs per visible (query, key) pair per head; under the causal
    mask query i sees Nk - Nq + i + 1 keys."""
    if w.causal:
        pairs = w.Nq * (w.Nk - w.Nq) + w.Nq * (w.Nq + 1) // 2
    else:
        pairs = w.Nq * w.Nk
    return 4.0 * w.B * w.Hq * w.d * pairs


def decode_min_bytes(w: DecodeWorkload) -> int:
    """K and V read once, Q read and O written once (bf16), lse written (fp32)."""
    kv = 2 * w.B * w.Nk * w.Hkv * w.d * 2
    qo = 2 * w.B * w.Nq * w.Hq * w.d * 2
    return kv + qo + 4 * w.B * w.Hq * w.Nq


def block_sparse_mask(Hq: int, N: int, seed: int, window: int = 2, density: float = 0.1):
    """A synthetic block mask [Hq, nb, nb] (uint8, nb = ceil(N / 128)): per
    head, a local window of query block i +- `window` key blocks, key block 0
    (every query sees the first tokens), and each other block with probability
    `density`, drawn from the seed."""
    nb = (N + 127) // 128
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    i = torch.arange(nb)
    local = (i[:, None] - i[None, :]).abs() <= window
    m = torch.rand((Hq, nb, nb), generator=g) < density
    m |= local
    m[:, :, 0] = True
    return m.to(torch.uint8)


def block_sparse_flops(mask, N: int, d: int, B: int, causal: bool) -> float:
    """FLOPs of the 128 x 128 blocks the kernel computes (QK^T and PV, 4 * 128
    * 128 * d each, ragged edge blocks at their true size), summed over heads
    and the batch; under the causal mask blocks above the diagonal are skipped
    and diagonal blocks count in full, as they are computed."""
    nb = (N + 127) // 128
    rows = torch.tensor([min(128, N - 128 * x) for x in range(nb)], dtype=torch.float64)
    m = mask.to(torch.float64)
    if causal:
        m = m * torch.tril(torch.ones(nb, nb, dtype=torch.float64))
    return float(4.0 * d * B * (m * rows[:, None] * rows[None, :]).sum())


def describe(w: Workload) -> str:
    return (f"B{w.B} Hq{w.Hq} Hkv{w.Hkv} N{w.N} d{w.d} "
            f"{'causal' if w.causal else 'non-causal'} scale={w.scale:.6g}")


def make_inputs(w: Workload, with_dout: bool = True):
    """Returns dict q, k, v[, dout] of bf16 CPU tensors, [B, N, H, d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = torch.randn((w.B, w.N, w.Hq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.N, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.N, w.Hkv, w.d), generator=g, dtype=torch.float32)
    if w.value_scale != 1.0:
        q.mul_(w.value_scale)
        k.mul_(w.value_scale)
        v.mul_(w.value_scale)
    if w.peaked_frac > 0.0:
        # ceil(frac * N) distinct key positions per (batch, kv head), drawn
        # without replacement from the same generator.
        npk = int(math.ceil(w.peaked_frac * w.N))
        for b in range(w.B):
            for h in range(w.Hkv):
                idx = torch.randperm(w.N, generator=g)[:npk]
                k[b, idx, h, :] *= w.peaked_mult
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    del q, k, v
    if with_dout:
        do = torch.randn((w.B, w.N, w.Hq, w.d), generator=g, dtype=torch.float32)
        out["dout"] = do.to(torch.bfloat16)
    return out


def peaked_positions(w: Workload):
    """The K rows made peaked by make_inputs, as {(b, h): LongTensor}."""
    if w.peaked_frac <= 0.0:
        return {}
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    # replay the draws in make_inputs' order
    torch.randn((w.B, w.N, w.Hq, w.d), generator=g)
    torch.randn((w.B, w.N, w.Hkv, w.d), generator=g)
    torch.randn((w.B, w.N, w.Hkv, w.d), generator=g)
    npk = int(math.ceil(w.peaked_frac * w.N))
    res = {}
    for b in range(w.B):
        for h in range(w.Hkv):
            res[(b, h)] = torch.randperm(w.N, generator=g)[:npk]
    return res


# ----------------------------------------------------------------------------
# accounting (nominal work and algorithmic bytes; no attention arithmetic)
# ----------------------------------------------------------------------------

def fwd_flops(w: Workload) -> float:
    """Nominal forward FLOPs: 4 * B * Hq * N^2 * d, halved under the causal mask."""
    f = 4.0 * w.B * w.Hq * w.N * w.N * w.d
    return f / 2 if w.causal else f


def bwd_flops(w: Workload) -> float:
    """Nominal backward FLOPs: 2.5 x the forward's."""
    return 2.5 * fwd_flops(w)


def fwd_min_bytes(w: Workload) -> int:
    """Q, K, V read once, O written once (bf16) and the fp32 row statistic."""
    qo = 2 * w.B * w.N * w.Hq * w.d * 2
    kv = 2 * w.B * w.N * w.Hkv * w.d * 2
    return qo + kv + 4 * w.B * w.Hq * w.N


def bwd_min_bytes(w: Workload) -> int:
    """Read Q, K, V, O, dO, lse; write dQ, dK, dV; D written and read once."""
    q_like = w.B * w.N * w.Hq * w.d * 2
    kv_like = w.B * w.N * w.Hkv * w.d * 2
    stats = 4 * w.B * w.Hq * w.N
    return 3 * q_like + 2 * kv_like + stats + q_like + 2 * kv_like + 2 * stats


def score_matrix_elements(N: int) -> int:
    """Entries of one head's N x N score matrix."""
    return N * N


def score_matrix_bytes(N: int, elem_bytes: int = 2) -> int:
    return score_matrix_elements(N) * elem_bytes
