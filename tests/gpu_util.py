"""Helpers for the GPU parity tests: guard-banded device buffers and bit checks."""
from __future__ import annotations

import numpy as np
import torch

SENTINEL = 0x7FC0DEAD  # a NaN bit pattern no fold of the test data produces
GUARD = 64             # elements of guard band on each side (256 bytes keeps the phase)


class Guarded:
    """A device f32 region of n elements at `offset` elements past a 256-byte
    boundary, with sentinel-filled guard bands before and after."""

    def __init__(self, n: int, offset: int = 0, fill: np.ndarray | None = None, device="cuda"):
        self.n, self.offset = n, offset
        self.buf = torch.empty(GUARD + offset + n + GUARD, dtype=torch.float32, device=device)
        self.buf.view(torch.int32).fill_(SENTINEL)
        self.lo = GUARD + offset
        self.t = self.buf[self.lo:self.lo + n]
        if fill is not None:
            self.t.copy_(torch.from_numpy(np.ascontiguousarray(fill, dtype=np.float32)).reshape(-1))

    def host(self) -> np.ndarray:
        return self.t.cpu().numpy()

    def intact(self) -> bool:
        b = self.buf.view(torch.int32)
        return bool((b[:self.lo] == SENTINEL).all() and (b[self.lo + self.n:] == SENTINEL).all())


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_bitwise(got: np.ndarray, want: np.ndarray, what: str) -> None:
    g, w = bits(got), bits(want)
    assert g.shape == w.shape, what
    bad = np.nonzero(g != w)[0]
    if bad.size:
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} of {g.size} words differ; first at {i}: "
                             f"got {g[i]:08x} want {w[i]:08x}")


def nonvacuous(a: np.ndarray) -> tuple[int, float]:
    """Nonzero count and absmax; an all-zero result proves nothing."""
    nz = int(np.count_nonzero(a))
    am = float(np.max(np.abs(a))) if a.size else 0.0
    return nz, am
