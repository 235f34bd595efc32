"""Guard canaries around the buffers the library writes.

compute-sanitizer is not available on the GPUs these tests run on, so bounds
are checked by construction: every output or workspace buffer a parity test
hands to the library sits inside a larger allocation whose bytes before and
after it (1 MiB each side, more than any tile or row-past-the-end store
could reach) hold a fixed byte pattern.  After the launch the test checks
that no byte of either guard changed.  The buffer itself starts NaN-filled
(outputs), so an element that is never written fails the parity check, and
a write past either end fails the guard check.
"""
from __future__ import annotations

import torch

GUARD_BYTES = 1 << 20
PATTERN = 0xA5  # 0xA5A5 is neither a plausible bf16 output nor a NaN


class Guarded:
    """A tensor of `shape` and `dtype` on `device` between two guard regions.
    `t` is the tensor (contiguous, 256-byte aligned); `check()` raises if a
    guard byte changed."""

    def __init__(self, shape, dtype, device, fill=float("nan")):
        numel = 1
        for s in shape:
            numel *= int(s)
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = numel * esize
        self.raw = torch.full((2 * GUARD_BYTES + self.nbytes,), PATTERN, dtype=torch.uint8,
                              device=device)
        inner = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes]
        self.t = inner.view(dtype).view(tuple(shape))
        if fill is not None and numel:
            self.t.fill_(fill)
        assert self.t.data_ptr() % 256 == 0

    def check(self, name: str = "buffer"):
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        for side, g in (("before", head), ("after", tail)):
            bad = (g != PATTERN).nonzero()
            assert bad.numel() == 0, (
                f"{name}: {bad.numel()} guard byte(s) {side} the buffer overwritten "
                f"(first at offset {int(bad[0]) - (GUARD_BYTES if side == 'before' else 0)}"
                f" {'from the start' if side == 'before' else 'past the end'})")


def guarded_like(t: torch.Tensor, fill=float("nan")) -> Guarded:
    return Guarded(t.shape, t.dtype, t.device, fill)


def check_all(**bufs):
    for name, g in bufs.items():
        if g is not None:
            g.check(name)
