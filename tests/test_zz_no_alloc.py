"""The allocation-free staged all-reduce against the existing staged entry point.

Some callers cannot call cudaMalloc: code running while a stream is captured
into a CUDA graph, and runtimes whose device memory is owned by their own
allocator or fixed up front. For them the library keeps its scratch in a
static device array (DETFOLD_NOALLOC_SCRATCH_BYTES) and the caller passes only
the arenas. These tests check, through the C ABI, that it gives the same bits
as detfold_loopback_allreduce_staged_ex with a caller workspace, on two calls in
a row (the second call reuses the scratch the first one left behind), and
that a request too large for the scratch is refused without running.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import detfold_inputs as gen
from gpu_util import Guarded, assert_bitwise

import deterministic_fixed_order_gb300 as df

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.mark.parametrize("W,n", [(2, 4096), (4, 65536 + 3), (3, (1 << 20) + 7), (6, 100_003)])
@pytest.mark.parametrize("flags", [0, 3])
def test_noalloc_matches_staged_with_caller_workspace(W, n, flags):
    rows = gen.normal_rows(W, n)
    scale = float(np.float32(1.0) / np.float32(W))
    ref = [Guarded(n, 0, rows[r]) for r in range(W)]
    new = [Guarded(n, r % 4, rows[r]) for r in range(W)]
    nb = df.detfold_staged_workspace_bytes(n, W)
    assert nb <= df.DETFOLD_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(nb // 4, dtype=torch.float32, device="cuda")
    for call in range(2):
        df.detfold_loopback_allreduce_staged_ex([a.t for a in ref], W, n, scale, flags, ws, nb)
        df.detfold_loopback_allreduce_staged_noalloc([a.t for a in new], W, n, scale, flags)
        torch.cuda.synchronize()
        for r in range(W):
            assert_bitwise(new[r].host(), ref[r].host(), f"W={W} n={n} call={call} rank={r}")
        assert all(a.intact() for a in ref + new)


def test_noalloc_refuses_requests_beyond_its_scratch():
    W = 4
    n = df.DETFOLD_NOALLOC_SCRATCH_BYTES // 4  # whole arenas of 16 MiB: the stack needs more
    assert df.detfold_staged_workspace_bytes(n, W) > df.DETFOLD_NOALLOC_SCRATCH_BYTES
    arenas = [torch.full((n,), float(r + 1), device="cuda") for r in range(W)]
    rc = df.status_loopback_allreduce_staged_noalloc([a for a in arenas], W, n, 1.0, 0)
    assert rc == df.STATUS["DETFOLD_ERR_SCRATCH_LIMIT"]
    torch.cuda.synchronize()
    for r in range(W):
        assert bool((arenas[r] == float(r + 1)).all())  # nothing ran
