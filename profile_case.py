"""Run one fold row at a chosen size for a few launches (for profiler captures).

    python profile_case.py ROW --len N [--W W] [--launches K] [--offset E]

ROW is one of: stacked, ptrs, allreduce, staged, scale, small, or torch_add
(torch's own elementwise add of two operands, W = 2, as a reference for a
launch of the same size that this library does not run). Inputs are
seeded synthetic data. --offset E starts every operand E elements past an
allocation boundary (E = 1 is the odd-world stress layout, base + 4 bytes;
stacked keeps its rows contiguous after the offset); --mixed adds 3r mod 8
elements to operand r, so every rank sits at its own 4-byte phase. Parity of these calls is
established by the test suite; this runner only launches them and reports
the status.
"""
from __future__ import annotations

import argparse
import os
import sys

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("row", choices=["stacked", "ptrs", "allreduce", "staged", "scale", "small", "torch_add"])
    ap.add_argument("--len", type=int, required=True)
    ap.add_argument("--W", type=int, default=8)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--offset", type=int, default=0)
    ap.add_argument("--mixed", action="store_true",
                    help="operand r at offset + (3r mod 8) elements: every rank at its own 4-byte phase")
    a = ap.parse_args()
    if not 0 <= a.offset < 64:
        ap.error("--offset must be in [0, 64)")

    import torch

    import deterministic_fixed_order_gb300 as df
    import detfold_inputs as gen

    dev = torch.device("cuda:0")
    W, n, off = a.W, a.len, a.offset
    rows = gen.gradient_rows(W, n)
    if a.row in ("stacked", "small"):
        flat = torch.empty(W * n + off, dtype=torch.float32, device=dev)
        d = flat[off:].view(W, n)
        d.copy_(torch.from_numpy(rows))
    else:  # one allocation per operand, each at the offset (plus its own phase with --mixed)
        shift = [(3 * r) % 8 if a.mixed else 0 for r in range(W)]
        d = [torch.empty(n + off + 8, dtype=torch.float32, device=dev)[off + shift[r]:off + shift[r] + n]
             for r in range(W)]
        for r in range(W):
            d[r].copy_(torch.from_numpy(rows[r]))
    out = torch.empty(n + off, dtype=torch.float32, device=dev)[off:]
    if a.row in ("stacked", "small"):
        fn = lambda: df.detfold_sum_stacked(out, d, W, n)
    elif a.row == "ptrs":
        srcs = [d[r] for r in range(W)]
        fn = lambda: df.detfold_sum_ptrs(out, srcs, W, n)
    elif a.row == "torch_add":  # reference: torch's own elementwise kernel on the same operands (W = 2)
        fn = lambda: torch.add(d[0], d[1], out=out)
    elif a.row == "scale":
        out.copy_(d[0])
        fn = lambda: df.detfold_scale(out, n, 0.5)
    else:
        arenas = [d[r] for r in range(W)]
        if a.row == "allreduce":
            fn = lambda: df.detfold_loopback_allreduce(arenas, W, n, 0.25)
        else:
            nb = df.detfold_staged_workspace_bytes(n, W)
            ws = torch.empty(nb // 4, dtype=torch.float32, device=dev)
            fn = lambda: df.detfold_loopback_allreduce_staged(arenas, W, n, 0.25, ws, nb)
    for _ in range(a.launches):
        fn()
    torch.cuda.synchronize()
    print(f"profile_case {a.row} W={W} len={n}: {a.launches} launches ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
