"""Writes tests/golden/c_client_case.txt: the expected outputs of the plain
C client's GPU mode (tests/c_client.c), computed by the float64 oracle only.

The inputs are not stored: the client and this script draw them from the same
counter-based generator, SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), each from its own
implementation.  Element i of tensor number t is
    u = splitmix64(t * 2^32 + i) >> 40          (24 bits)
    x = (u - 2^23) / 2^23                        (exact in float32)
rounded to bf16 to nearest, ties to even.  The file holds, per output tensor,
its float64 L2 norm and the exact values at a fixed set of sampled flat
indices (every row of the ragged last tile among them).

Run:  python tests/golden/make_c_client_case.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

B, H, HKV, N, D, CAUSAL, SCALE = 1, 2, 1, 200, 64, 1, 0.125
MASK64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    z = (x + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def bf16_round(x32: np.ndarray) -> np.ndarray:
    """float32 -> the nearest bf16 (ties to even), returned as float64."""
    b = x32.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def tensor(t: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    u = np.array([splitmix64((t << 32) + i) >> 40 for i in range(n)], dtype=np.int64)
    x = ((u - (1 << 23)) / float(1 << 23)).astype(np.float32)
    return bf16_round(x).reshape(shape)


def main():
    q = tensor(0, (B, N, H, D))
    k = tensor(1, (B, N, HKV, D))
    v = tensor(2, (B, N, HKV, D))
    do = tensor(3, (B, N, H, D))
    o, lse = oracle.attn_fwd(q, k, v, bool(CAUSAL), SCALE)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, bool(CAUSAL), SCALE)
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c_client_case.txt")
    with open(out, "w") as f:
        f.write("# expected outputs for tests/c_client.c (written by make_c_client_case.py)\n")
        f.write(f"shape {B} {H} {HKV} {N} {D} {CAUSAL} {SCALE!r}\n")
        for name, arr in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
            flat = arr.ravel()
            f.write(f"norm {name} {np.linalg.norm(flat):.17g}\n")
            # every 97th element, and every element of the ragged last rows
            idx = set(range(0, flat.size, 97))
            if name == "lse":
                idx |= {h * N + i for h in range(H) for i in range(128, N)}
            else:
                width = arr.shape[2] * arr.shape[3]
                idx |= {i * width + c for i in range(N - 2, N) for c in range(width)}
            for i in sorted(idx):
                f.write(f"{name} {i} {flat[i]:.17g}\n")
    print(out)


if __name__ == "__main__":
    main()
