"""Benchmark of the fixed-order fold hot path on GB300.

One step = one pass over every row of the hot path at its workload size:

  c3_stacked  W=8 stacked [8][2^26] f32 fold, gradient-like values (2 GiB in)
  c3_ptrs     the same rows through the pointer-table fold
  c4_fused    fused loopback all-reduce, W=4 arenas of 1e8 f32, x0.25 mean
  c4_staged   the reference's own dataflow (exchange + fold + distribute)
              on a second set of W=4 x 1e8 arenas, same mean
  c5_w3/c5_w6 odd worlds, len 2^20+7 at base+4 bytes, stress values:
              pointer-table sum, the mean as its own pass, fused all-reduce
  c2_16k/256k W=2 decode-join folds (n = 4096 and 65536) on the small path

`value` = algorithmic bytes of the step / device time of the step (GB/s),
inputs resident in HBM. Algorithmic bytes per call: (W+1)*len*4 for a sum,
2*len*4 for the mean pass, 2*W*len*4 for an all-reduce (the staged
comparator is charged the same algorithmic bytes although it moves
(4W+1)*len*4: exchange 2W, fold W+1, distribute W). The step reads and writes ~11 GB, far more than the 129 MB
L2, so no L2 flush is needed between steps.

Also reported: per-row kernel times from CUDA events on the launching
stream, the roofline of the dominant kernel, microseconds per call of the
16 KiB W=2 fold inside a 10,000-node CUDA graph (with the empty-kernel,
the one-warp memory round-trip and the same-launch-shape floors of
libdetfold_probes), an end-to-end figure through the public API with host buffers, SM
clocks sampled during the run, a sampled bit-exact check of the bench's own
outputs against the CPU oracle, and the oracle timed on host cores.

`--impl reference` times the CPU oracle instead (on bounded samples of the
same workload), the program the fold is checked against.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fold effective HBM GB/s and % of GB300 peak; µs/call at 16 KiB W=2"
FALLBACK_HBM_GBS = 6800.0

C3_W, C3_N = 8, 1 << 26
C4_W, C4_N = 4, 100_000_000
C5_N = (1 << 20) + 7
C5_WS = (3, 6)
C2_NS = (4096, 65536)
GRAPH_NODES = 10_000
E2E_PASSES = 5  # end-to-end passes; `e2e.value` is their median

# DRAM traffic of the dominant kernel from one ncu capture, keyed by a hash of
# the kernel sources it was taken on; null once the kernel has changed.
NCU_TRAFFIC = {
    # profiles/fold_bulk_kernel_W8_sum.md: full-size C3 launch (8 x 2^26),
    # dram__bytes_read.sum + dram__bytes_write.sum
    "fold_bulk_kernel<W=8,sum>": {"bytes_per_launch": 2147553536 + 259127552,
                                  "kernel_hash": "189637e941c52b05"},
    # profiles/fold_bulk_kernel_W4_allreduce.md: full-size C4 launch (4 x 1e8)
    "fold_bulk_kernel<W=4,all-reduce>": {"bytes_per_launch": 1600032000 + 1538591744,
                                         "kernel_hash": "189637e941c52b05"},
}

KERNEL_FILES = ("detfold_kernels.cuh", "detfold_launch.cuh", "detfold_async.cuh", "fold_sum_nc.cu",
                "fold_sum_coherent.cu", "fold_allreduce.cu", "fold_bulk.cu", "fold_table.cu",
                "move_kernels.cu", "one_shot.cu")


def _code_only(text: str) -> str:
    """C++ source without comments or whitespace: what a capture depends on."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_source_hash() -> str:
    """Hash of every kernel source and its launch configuration (code only:
    editing a comment does not invalidate a profile)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "deterministic_fixed_order_gb300", "csrc")
    for f in KERNEL_FILES:
        with open(os.path.join(csrc, f)) as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def row_bytes() -> dict[str, int]:
    b = {
        "c3_stacked": (C3_W + 1) * C3_N * 4,
        "c3_ptrs": (C3_W + 1) * C3_N * 4,
        "c4_fused": 2 * C4_W * C4_N * 4,
        "c4_staged": 2 * C4_W * C4_N * 4,
    }
    for W in C5_WS:
        b[f"c5_w{W}"] = ((W + 1) + 2 + 2 * W) * C5_N * 4
    for n in C2_NS:
        b[f"c2_{n}"] = 3 * n * 4
    return b


def step_input_bytes() -> int:
    """Bytes of a step's distinct host inputs: the C3 stack, the C4 arenas,
    the C5 rows and the C2 rows, each counted once."""
    return 4 * (C3_W * C3_N + C4_W * C4_N + sum(W * C5_N for W in C5_WS) + sum(2 * n for n in C2_NS))


def peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if k in d and d[k]:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time: every rank runs its own replica, the job is
    done when the last one is."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, step_bytes: int, ms_per_step: float) -> float:
    """All ranks' algorithmic bytes over the slowest rank's step time."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="detfold_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0: float | None = None):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[4:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for name, v in zip(names[1:], flags[1:]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        loaded = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU arm

class Workload:
    """Device buffers of one step, generated on the host and copied once."""

    def __init__(self, torch, df, gen, dev):
        self.torch, self.df, self.dev = torch, df, dev
        t = torch
        pin = lambda n: t.empty(n, dtype=t.float32, pin_memory=True)
        # host inputs (pinned: also the sources of the end-to-end leg)
        self.h_c3 = pin(C3_W * C3_N)
        gen.fill_recipe("gradient", self.h_c3.data_ptr(), C3_W, C3_N, C3_N)
        self.h_c4 = pin(C4_W * C4_N)
        gen.fill_recipe("normal", self.h_c4.data_ptr(), C4_W, C4_N, C4_N)
        self.h_c5 = {}
        for W in C5_WS:
            h = pin(W * C5_N)
            gen.fill_recipe("stress", h.data_ptr(), W, C5_N, C5_N)
            self.h_c5[W] = h
        self.h_c2 = {}
        for n in C2_NS:
            h = pin(2 * n)
            gen.fill_recipe("vecf", h.data_ptr(), 2, n, n)
            self.h_c2[n] = h
        self._device_buffers()
        self.scale4 = df.detfold_mean_scale(C4_W)
        self.scale5 = {W: df.detfold_mean_scale(W) for W in C5_WS}
        torch.cuda.synchronize()

    def device_twin(self):
        """The same workload (the same host inputs) on a second set of device
        buffers: the end-to-end leg alternates steps between the two sets."""
        import copy
        twin = copy.copy(self)
        twin._device_buffers()
        self.torch.cuda.synchronize()
        return twin

    def _device_buffers(self):
        t, dev, df = self.torch, self.dev, self.df
        self.c3 = self.h_c3.to(dev)
        self.c3_rows = [self.c3[r * C3_N:(r + 1) * C3_N] for r in range(C3_W)]
        self.c3_out = t.empty(C3_N, dtype=t.float32, device=dev)
        self.c3_out2 = t.empty(C3_N, dtype=t.float32, device=dev)
        self.c4f = [self.h_c4[r * C4_N:(r + 1) * C4_N].to(dev) for r in range(C4_W)]
        self.c4s = [self.h_c4[r * C4_N:(r + 1) * C4_N].to(dev) for r in range(C4_W)]
        self.ws_bytes = df.detfold_staged_workspace_bytes(C4_N, C4_W)
        self.ws = t.empty(self.ws_bytes // 4, dtype=t.float32, device=dev)
        # C5: every arena at base + 4 bytes (one element past a 512-byte boundary)
        self.c5_buf, self.c5_sum_src, self.c5_ar, self.c5_out = {}, {}, {}, {}
        for W in C5_WS:
            self.c5_sum_src[W] = []
            self.c5_ar[W] = []
            keep = []
            for r in range(W):
                for dst in (self.c5_sum_src[W], self.c5_ar[W]):
                    b = t.empty(C5_N + 1, dtype=t.float32, device=dev)
                    v = b[1:1 + C5_N]
                    v.copy_(self.h_c5[W][r * C5_N:(r + 1) * C5_N])
                    keep.append(b)
                    dst.append(v)
            ob = t.empty(C5_N + 1, dtype=t.float32, device=dev)
            keep.append(ob)
            self.c5_out[W] = ob[1:1 + C5_N]
            self.c5_buf[W] = keep
        self.c2 = {n: self.h_c2[n].to(dev) for n in C2_NS}
        self.c2_out = {n: t.empty(n, dtype=t.float32, device=dev) for n in C2_NS}

    def rows(self):
        """(name, callable, kernel launches) in step order."""
        df = self.df
        out = [
            ("c3_stacked", lambda: df.detfold_sum_stacked(self.c3_out, self.c3, C3_W, C3_N), 1),
            ("c3_ptrs", lambda: df.detfold_sum_ptrs(self.c3_out2, self.c3_rows, C3_W, C3_N), 1),
            ("c4_fused", lambda: df.detfold_loopback_allreduce(self.c4f, C4_W, C4_N, self.scale4), 1),
            ("c4_staged", lambda: df.detfold_loopback_allreduce_staged(
                self.c4s, C4_W, C4_N, self.scale4, self.ws, self.ws_bytes), 3 * C4_W),
        ]
        for W in C5_WS:
            def c5(W=W):
                df.detfold_sum_ptrs(self.c5_out[W], self.c5_sum_src[W], W, C5_N)
                df.detfold_scale(self.c5_out[W], C5_N, self.scale5[W])
                df.detfold_loopback_allreduce(self.c5_ar[W], W, C5_N, self.scale5[W])
            out.append((f"c5_w{W}", c5, 3))
        for n in C2_NS:
            out.append((f"c2_{n}", lambda n=n: df.detfold_sum_stacked(self.c2_out[n], self.c2[n], 2, n), 1))
        return out


def collect_step_samples(wl, steps_run: int, rng) -> list[dict]:
    """Host copies of the bench's own outputs on sampled columns, with the
    host inputs those columns came from (no oracle here: `verify_samples`, in
    the oracle leg, computes what they must be). The all-reduces are in place,
    so after k steps their state is k repeated all-reduces."""
    specs = []
    idx3 = np.sort(rng.choice(C3_N, 4096, replace=False))
    rows3 = np.ascontiguousarray(wl.h_c3.numpy().reshape(C3_W, C3_N)[:, idx3])
    specs.append({"group": "c3", "kind": "fold_stacked", "inputs": rows3,
                  "got": [wl.c3_out.cpu().numpy()[idx3], wl.c3_out2.cpu().numpy()[idx3]]})
    idx4 = np.sort(rng.choice(C4_N, 4096, replace=False))
    h4 = wl.h_c4.numpy().reshape(C4_W, C4_N)
    specs.append({"group": "c4", "kind": "allreduce", "repeat": steps_run, "scale": wl.scale4,
                  "inputs": [np.ascontiguousarray(h4[r, idx4]) for r in range(C4_W)],
                  "got": [[wl.c4f[r].cpu().numpy()[idx4] for r in range(C4_W)],
                          [wl.c4s[r].cpu().numpy()[idx4] for r in range(C4_W)]]})
    for W in C5_WS:
        h5 = wl.h_c5[W].numpy().reshape(W, C5_N)
        idx5 = np.r_[0:16, np.sort(rng.choice(np.arange(16, C5_N), 2048, replace=False))]
        cols = np.ascontiguousarray(h5[:, idx5])
        specs.append({"group": "c5", "kind": "fold_scale", "inputs": cols, "scale": wl.scale5[W],
                      "got": [wl.c5_out[W].cpu().numpy()[idx5]]})
        specs.append({"group": "c5", "kind": "allreduce", "repeat": steps_run, "scale": wl.scale5[W],
                      "inputs": [np.ascontiguousarray(cols[r]) for r in range(W)],
                      "got": [[wl.c5_ar[W][r].cpu().numpy()[idx5] for r in range(W)]]})
    for n in C2_NS:
        specs.append({"group": "c2", "kind": "fold_stacked", "inputs": wl.h_c2[n].numpy().reshape(2, n),
                      "got": [wl.c2_out[n].cpu().numpy()]})
    return specs


def verify_samples(oracle, specs: list[dict]) -> dict:
    """Words that differ from the oracle, by group, for collected samples."""
    res = {}
    for sp in specs:
        if sp["kind"] == "fold_stacked":
            want = [oracle.fold_stacked(sp["inputs"])]
            gots = [[g] for g in sp["got"]]
        elif sp["kind"] == "fold_scale":
            want = [oracle.scale(oracle.fold(sp["inputs"]), np.float32(sp["scale"]))]
            gots = [[g] for g in sp["got"]]
        else:  # allreduce, repeated
            want = [a.copy() for a in sp["inputs"]]
            for _ in range(sp["repeat"]):
                oracle.allreduce(want, np.float32(sp["scale"]))
            gots = sp["got"]
        d = sum(oracle.bit_diffs(g, w) for got in gots for g, w in zip(got, want))
        res[sp["group"]] = res.get(sp["group"], 0) + int(d)
    return res


PROBES_LIB = os.path.join(ROOT, "deterministic_fixed_order_gb300", "libdetfold_probes.so")


class Probes:
    """The latency-floor kernels of libdetfold_probes.so (include/detfold_probes.h),
    a measurement library of its own that the fold library never loads."""

    def __init__(self, path: str = PROBES_LIB):
        import ctypes
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        self.lib = lib = ctypes.CDLL(path)
        lib.detfold_probe_launch_floor.argtypes = [I, I, P]
        lib.detfold_probe_memory_floor.argtypes = [P, P, I, I, P]
        lib.detfold_probe_same_shape_floor.argtypes = [P, P, P, I64, I, P]
        for name in ("detfold_probe_launch_floor", "detfold_probe_memory_floor",
                     "detfold_probe_same_shape_floor", "detfold_probe_last_cuda_error"):
            getattr(lib, name).restype = I

    @staticmethod
    def _stream(stream) -> int:
        import torch
        return (stream or torch.cuda.current_stream()).cuda_stream

    def _check(self, rc: int, where: str) -> None:
        if rc != 0:
            raise RuntimeError(f"{where}: status {rc} (cudaError {self.lib.detfold_probe_last_cuda_error()})")

    def launch_floor(self, count: int, pdl: int = 1, stream=None) -> None:
        self._check(self.lib.detfold_probe_launch_floor(count, pdl, self._stream(stream)), "launch_floor")

    def memory_floor(self, src, dst, count: int, pdl: int = 1, stream=None) -> None:
        self._check(self.lib.detfold_probe_memory_floor(src.data_ptr(), dst.data_ptr(), count, pdl,
                                                        self._stream(stream)), "memory_floor")

    def same_shape_floor(self, out, src0, src1, n: int, count: int, stream=None) -> None:
        self._check(self.lib.detfold_probe_same_shape_floor(out.data_ptr(), src0.data_ptr(), src1.data_ptr(),
                                                            n, count, self._stream(stream)),
                    "same_shape_floor")


def graph_us_per_call(torch, df, wl, rounds: int = 5, reps: int = 5) -> dict:
    """Microseconds per call of graphs of GRAPH_NODES back-to-back calls: the
    W=2 fold at each C2 size (pointer table in the kernel parameters, and
    through a device-resident table), beside the floors of libdetfold_probes
    -- an empty kernel with and without programmatic dependent launch, a
    one-warp load-after-predecessor + store, and at each C2 size a kernel of
    the fold's own launch shape that moves the same bytes without the adds.
    Every graph is captured first and then timed round-robin (`rounds` x
    `reps` replays each), so a drift of the GPU's state during the section
    shifts all of them alike; each figure is the median over its replays."""
    probes = Probes()
    stream = torch.cuda.Stream()

    def capture(fn):
        with torch.cuda.stream(stream):
            fn()  # first use outside the capture
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        return g

    def rep(fn):
        return lambda: [fn() for _ in range(GRAPH_NODES)]

    graphs, keep = {}, []
    for n in C2_NS:
        graphs[(str(n), "us_per_call")] = capture(rep(lambda n=n: df.detfold_sum_stacked(
            wl.c2_out[n], wl.c2[n], 2, n)))
        table = df.device_table([wl.c2[n][:n], wl.c2[n][n:]])
        keep.append(table)
        graphs[(str(n), "us_per_call_device_table")] = capture(rep(lambda n=n, table=table: df.detfold_sum_ptrs_dev(
            wl.c2_out[n], table, 2, n)))
        so = torch.empty(n, dtype=torch.float32, device=wl.dev)
        keep.append(so)
        graphs[(str(n), "same_shape_floor_us")] = capture(lambda n=n, so=so: probes.same_shape_floor(
            so, wl.c2[n][:n], wl.c2[n][n:], n, GRAPH_NODES))
    pair = torch.zeros(64, device="cuda")
    graphs[("floors", "empty_pdl")] = capture(lambda: probes.launch_floor(GRAPH_NODES, 1))
    graphs[("floors", "empty_plain")] = capture(lambda: probes.launch_floor(GRAPH_NODES, 0))
    graphs[("floors", "memory_pdl")] = capture(lambda: probes.memory_floor(pair[:32], pair[32:],
                                                                          GRAPH_NODES, 1))
    times = {k: [] for k in graphs}
    for _ in range(rounds):
        for k, g in graphs.items():
            for _ in range(reps):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a.record()
                    g.replay()
                    b.record()
                b.synchronize()
                times[k].append(a.elapsed_time(b) * 1e3 / GRAPH_NODES)
    res = {}
    for (group, key), ts in times.items():
        res.setdefault(group, {})[key] = round(statistics.median(ts), 3)
    res["floors"]["spread_us"] = round(max(max(v) - min(v) for v in times.values()), 3)
    for n in C2_NS:
        r = res[str(n)]
        r["ratio_to_same_shape_floor"] = round(r["us_per_call"] / r["same_shape_floor_us"], 3)
        r["ratio_to_memory_floor"] = round(r["us_per_call"] / res["floors"]["memory_pdl"], 3)
        r["ratio_to_empty_floor"] = round(r["us_per_call"] / res["floors"]["empty_pdl"], 3)
    del graphs
    # the bits after all the replays must equal one fold: every word goes to
    # the oracle leg
    torch.cuda.synchronize()
    res["_specs"] = [{"group": f"c2_{n}_after_graph_replays", "kind": "fold_stacked",
                      "inputs": wl.h_c2[n].numpy().reshape(2, n), "got": [wl.c2_out[n].cpu().numpy()]}
                     for n in C2_NS]
    return res


def next_rows(torch, df, wl, reps: int = 10, calls: int = 5) -> dict:
    """Rows beyond the step: pure-movement broadcast and all-gather, the
    all-reduce at mixed phases, the realigned stack and the fold over a
    device-resident pointer table, in algorithmic GB/s. Every operand is
    larger than L2, and each row is timed as `calls` back-to-back calls
    between two events (ms per call, median of `reps`), so a figure is the
    row's streaming rate, not one call's launch and ramp."""
    def t(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(calls):
                fn()
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b) / calls)
        return statistics.median(ms)
    out = {}
    # broadcast: C3 row 0 to the other seven rows' worth of space (reads 1, writes 7)
    dsts = [torch.empty(C3_N, dtype=torch.float32, device=wl.dev) for _ in range(7)]
    ms = t(lambda: df.detfold_broadcast(dsts, 7, wl.c3_rows[0], C3_N))
    out["broadcast_1to7_2^26"] = {"ms": round(ms, 4), "gbs": round(8 * C3_N * 4 / (ms * 1e-3) / 1e9, 1)}
    del dsts
    span, W = 1 << 24, 4
    outs = [torch.empty(W * span, dtype=torch.float32, device=wl.dev) for _ in range(W)]
    parts = [wl.c3_rows[r][:span] for r in range(W)]
    ms = t(lambda: df.detfold_all_gather(outs, W, parts, span))
    out["all_gather_W4_2^24"] = {"ms": round(ms, 4),
                                 "gbs": round((W + W * W) * span * 4 / (ms * 1e-3) / 1e9, 1)}
    del outs
    # one-shot emulation at the decode-join size, per-call device time
    n = 4096
    arenas = [wl.c2[n][:n].clone(), wl.c2[n][n:].clone()]
    link = df.OneShotLink(2, n, device=wl.dev)

    def per_call_us(fn, calls=200):
        ts = []
        for _ in range(calls):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts)
    for _ in range(5):
        link.all_reduce(arenas)
    torch.cuda.synchronize()

    def one_shot():
        df.detfold_one_shot_allreduce(arenas, 2, n, 1.0, link.link, 0, link.stage, link.words)
    out["one_shot_W2_16KiB_us_per_call"] = round(per_call_us(one_shot), 2)
    out["one_shot_barrier_errors"] = link.barrier_errors()
    out["fused_W2_16KiB_us_per_call_same_timing"] = round(
        per_call_us(lambda: df.detfold_loopback_allreduce(arenas, 2, n, 1.0)), 2)
    # the same two calls back to back in CUDA graphs of 1000 nodes (the
    # one-shot takes each node's epoch from the link's counter)
    gs = torch.cuda.Stream()
    for key, fn in (("one_shot_W2_16KiB_graph_us_per_call", one_shot),
                    ("fused_W2_16KiB_graph_us_per_call",
                     lambda: df.detfold_loopback_allreduce(arenas, 2, n, 1.0))):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            for _ in range(1000):
                fn()
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(7):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(gs):
                a.record()
                g.replay()
                b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        out[key] = round(statistics.median(ts), 3)  # ms per 1000 calls = us per call
        del g
    out["one_shot_barrier_errors_after_graphs"] = link.barrier_errors()
    # the C5 rows (sum, mean pass, all-reduce) back to back in a graph of 100
    # rows: their device time without the per-row event records of the step
    row_fns = {name: fn for name, fn, _ in wl.rows()}
    rb = row_bytes()
    for W in C5_WS:
        key = f"c5_w{W}"
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            for _ in range(100):
                row_fns[key]()
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(7):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(gs):
                a.record()
                g.replay()
                b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b) / 100)
        ms = statistics.median(ts)
        out[f"{key}_graph"] = {"us": round(ms * 1e3, 2), "gbs": round(rb[key] / (ms * 1e-3) / 1e9, 1)}
        del g
    # mismatched phases at the C3 size: the rows of an [8][2^26 - 3] stack sit
    # at eight different 4-byte phases, so the realigned kernel runs
    nm = C3_N - 3
    ms = t(lambda: df.detfold_sum_stacked(wl.c3_out2, wl.c3, C3_W, nm))
    out["stacked_mismatched_W8_2^26-3"] = {"ms": round(ms, 4),
                                           "gbs": round((C3_W + 1) * nm * 4 / (ms * 1e-3) / 1e9, 1)}
    table = df.device_table(wl.c3_rows)
    ms = t(lambda: df.detfold_sum_ptrs_dev(wl.c3_out2, table, C3_W, C3_N))
    out["sum_ptrs_dev_W8_2^26"] = {"ms": round(ms, 4),
                                   "gbs": round((C3_W + 1) * C3_N * 4 / (ms * 1e-3) / 1e9, 1)}
    # the fused all-reduce with arenas at different 4-byte phases (realigned
    # loads and stores), 2^24 elements per arena: W=3 and 6 at the C5
    # per-rank phases 4*(r mod 4) bytes, W=4 at phases 0-3, W=8 at 4*(3r mod 8)
    n = 1 << 24
    bufs = [torch.empty(n + 8, dtype=torch.float32, device=wl.dev) for _ in range(8)]
    for W, phase in ((3, lambda r: r % 4), (4, lambda r: r), (6, lambda r: r % 4), (8, lambda r: (3 * r) % 8)):
        arenas = [bufs[r][phase(r):phase(r) + n] for r in range(W)]
        for a in arenas:
            a.normal_()
        m = df.detfold_mean_scale(W)
        ms = t(lambda: df.detfold_loopback_allreduce(arenas, W, n, m))
        out[f"allreduce_mixed_phase_W{W}_2^24"] = {
            "ms": round(ms, 4), "gbs": round(2 * W * n * 4 / (ms * 1e-3) / 1e9, 1),
            "phases_bytes": [4 * phase(r) for r in range(W)]}
    del bufs
    out["timing"] = f"the large rows: {calls} back-to-back calls per event pair, median of {reps}"
    return out


def c5_launches(torch, df, wl, sets: int = 12, reps: int = 4, rounds: int = 2) -> dict:
    """Device time per launch at the C5 length (2^20+7 at base + 4 B), each
    of the row's three calls alone and the whole row (the three in order),
    beside torch's own elementwise kernels at the same length (an add of two
    rows into a third; an in-place multiply of one row). Each figure comes from a CUDA graph of `reps` x `sets`
    back-to-back launches over `sets` buffer sets whose footprint exceeds L2,
    so every launch reads cold data but none pays a host launch; median of 9
    replays, the best of `rounds` interleaved rounds. At this length a
    launch's fixed cost (the predecessor's retirement, the first DRAM round
    trip, the ramp over the SMs) is comparable to its transfer time."""
    dev, n = wl.dev, C5_N
    stream = torch.cuda.Stream()

    def per_launch_us(enq):
        with torch.cuda.stream(stream):
            for k in range(sets):
                enq(k)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                for k in range(sets):
                    enq(k)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(9):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record()
                g.replay()
                b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / (reps * sets))
        del g
        return statistics.median(ts)

    calls, nbytes = {}, {}
    for W in C5_WS:
        bufs = []
        for k in range(sets):
            b = torch.empty((2 * W + 1, n + 1), dtype=torch.float32, device=dev)
            for r in range(W):
                b[r, 1:].copy_(wl.c5_sum_src[W][r])
                b[W + r, 1:].copy_(wl.c5_sum_src[W][r])
            bufs.append(([b[r, 1:] for r in range(W)], [b[W + r, 1:] for r in range(W)], b[2 * W, 1:]))
        m = wl.scale5[W]
        calls[f"w{W}_sum"] = lambda k, W=W, bufs=bufs: df.detfold_sum_ptrs(bufs[k][2], bufs[k][0], W, n)
        calls[f"w{W}_mean_pass"] = lambda k, bufs=bufs, m=m: df.detfold_scale(bufs[k][2], n, m)
        calls[f"w{W}_allreduce"] = lambda k, W=W, bufs=bufs, m=m: df.detfold_loopback_allreduce(
            bufs[k][1], W, n, m)
        nbytes[f"w{W}_sum"] = (W + 1) * n * 4
        nbytes[f"w{W}_mean_pass"] = 2 * n * 4
        nbytes[f"w{W}_allreduce"] = 2 * W * n * 4

        def row(k, W=W, bufs=bufs, m=m):  # the step's C5 row: the three calls in order
            df.detfold_sum_ptrs(bufs[k][2], bufs[k][0], W, n)
            df.detfold_scale(bufs[k][2], n, m)
            df.detfold_loopback_allreduce(bufs[k][1], W, n, m)
        calls[f"w{W}_row"] = row
        nbytes[f"w{W}_row"] = nbytes[f"w{W}_sum"] + nbytes[f"w{W}_mean_pass"] + nbytes[f"w{W}_allreduce"]
    tbufs = [torch.randn((3, n), device=dev) for _ in range(sets)]
    calls["torch_add"] = lambda k: torch.add(tbufs[k][0], tbufs[k][1], out=tbufs[k][2])
    calls["torch_mul_inplace"] = lambda k: tbufs[k][2].mul_(0.5)
    nbytes["torch_add"] = 3 * n * 4
    nbytes["torch_mul_inplace"] = 2 * n * 4
    best = {}
    for _ in range(rounds):
        for key, fn in calls.items():
            us = per_launch_us(fn)
            best[key] = min(best.get(key, us), us)
    peak, _ = peaks()
    out = {key: {"us": round(us, 3), "gbs": round(nbytes[key] / (us * 1e-6) / 1e9, 1),
                 "frac": round(nbytes[key] / (us * 1e-6) / 1e9 / peak, 4)}
           for key, us in best.items()}
    out["timing"] = (f"graphs of {reps} x {sets} launches over {sets} buffer sets (cold data), "
                     f"median of 9 replays, best of {rounds} rounds")
    return out


def arm_config(world: int) -> dict:
    """The workload both arms report: one pass of every hot-path row."""
    return {
        "workload": "one pass of every hot-path row: C3 W=8x2^26 stacked + ptrs fold, "
                    "C4 W=4x1e8 fused and staged loopback all-reduce x0.25, "
                    "C5 W=3,6 x (2^20+7) at base+4B sum/mean/all-reduce, "
                    "C2 W=2 n=4096 and 65536 small-path folds",
        "step_algorithmic_bytes": sum(row_bytes().values()),
        "l2": "inputs larger than L2 (~11 GB per step), no flush",
        "parallelism": f"replicas x{world} (one independent loopback world per GPU)",
    }


def host_link_gbs(torch, dev, reps: int = 5) -> dict:
    """Host<->device link rates in this run, best of `reps`: a 1 GiB copy from
    pinned host memory to the device, the reverse, and both at once on two
    streams (bytes of both directions / time)."""
    n = 1 << 28
    h_in = torch.empty(n, dtype=torch.float32, pin_memory=True)
    h_out = torch.empty(n, dtype=torch.float32, pin_memory=True)
    d_a = torch.empty(n, dtype=torch.float32, device=dev)
    d_b = torch.empty(n, dtype=torch.float32, device=dev)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def best(streams_and_fns, nbytes):
        top = 0.0
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for st, fn in streams_and_fns:
                with torch.cuda.stream(st):
                    fn()
            torch.cuda.synchronize()
            top = max(top, nbytes / (time.perf_counter() - t0) / 1e9)
        return top

    nb = n * 4
    res = {"h2d_gbs": best([(up, lambda: d_a.copy_(h_in, non_blocking=True))], nb),
           "d2h_gbs": best([(down, lambda: h_out.copy_(d_b, non_blocking=True))], nb),
           "both_gbs": best([(up, lambda: d_a.copy_(h_in, non_blocking=True)),
                             (down, lambda: h_out.copy_(d_b, non_blocking=True))], 2 * nb)}
    del h_in, h_out, d_a, d_b
    return res


class LinkSample:
    """A short both-ways sample of the host link (256 MiB each way on two
    streams, median of 3), taken right after each end-to-end pass, so that a
    slow pass can be set against the link's rate at that moment."""

    def __init__(self, torch, dev, n: int = 1 << 26):
        self.torch = torch
        self.h_in = torch.empty(n, dtype=torch.float32, pin_memory=True)
        self.h_out = torch.empty(n, dtype=torch.float32, pin_memory=True)
        self.d_a = torch.empty(n, dtype=torch.float32, device=dev)
        self.d_b = torch.empty(n, dtype=torch.float32, device=dev)
        self.up, self.down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        self.nbytes = 2 * n * 4

    def __call__(self, reps: int = 3) -> float:
        torch, ts = self.torch, []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            with torch.cuda.stream(self.up):
                self.d_a.copy_(self.h_in, non_blocking=True)
            with torch.cuda.stream(self.down):
                self.h_out.copy_(self.d_b, non_blocking=True)
            torch.cuda.synchronize()
            ts.append(self.nbytes / (time.perf_counter() - t0) / 1e9)
        return statistics.median(ts)


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, vendor figure (context only)


def copy_peak_gbs(torch, df, dev, reps: int = 20) -> dict:
    """Achievable 1:1 read/write bandwidth on this GPU in this run, best of
    `reps`: a 1 GiB device-to-device copy (torch copy_, a D2D memcpy) and
    this library's W=1 fold of 2^28 floats (a 1:1 stream kernel on the same
    bulk-async path as the folds), both charged 2 GiB per call."""
    a = torch.empty(1 << 28, dtype=torch.float32, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)

    def best(fn):
        fn()
        torch.cuda.synchronize()
        top = 0.0
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            top = max(top, 2 * a.numel() * 4 / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        return top

    res = {"d2d_copy_gbs": best(lambda: b.copy_(a)),
           "stream_kernel_gbs": best(lambda: df.detfold_sum_stacked(b, a, 1, a.numel()))}
    del a, b
    return res


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
        if m:
            return m.group(1).strip()
        part = re.search(r"^CPU part\s*:\s*(\S+)$", info, re.M)
        impl = re.search(r"^CPU implementer\s*:\s*(\S+)$", info, re.M)
        if part and impl:
            return f"implementer {impl.group(1)}, part {part.group(1)}"
    except OSError:
        pass
    return "unknown"


def oracle_leg(gen, world: int, samples: list[dict]) -> tuple[dict | None, dict]:
    """The bench's oracle leg, the one place the GPU arm uses the CPU oracle:
    it replays the oracle on the samples the GPU arm collected (words that
    differ, by group), and at N=1 times the oracle on host cores
    (cpu_baseline). The GPU arm itself never calls the oracle."""
    import oracle
    checks = verify_samples(oracle, samples)
    return (cpu_baseline(oracle, gen) if world == 1 else None), checks


def cpu_baseline(oracle, gen, budget_s: float = 12.0, split_budget_s: float = 4.0) -> dict:
    """The oracle as it stands on a bounded sample of every row of the step:
    the first S elements of each rank's arena (S = 2^21 for the large rows,
    the full length for the small ones), repeated until the budget is spent.
    `value` is single-threaded. `threads_split` is the same per-element chains
    with every row's elements split into one contiguous range per host core,
    each range folded by the same oracle call on its own thread (the oracle's
    C calls release the GIL); the chain of every element is unchanged."""
    S = 1 << 21
    c3 = gen.gradient_rows(C3_W, S)
    c4 = gen.normal_rows(C4_W, S)
    c5 = {W: gen.stress_rows(W, C5_N) for W in C5_WS}
    c2 = {n: gen.c1_rows(2, n) for n in C2_NS}
    s4 = np.float32(0.25)
    pass_bytes = (2 * (C3_W + 1) * S * 4 + 2 * (2 * C4_W * S * 4)
                  + sum(((W + 1) + 2 + 2 * W) * C5_N * 4 for W in C5_WS)
                  + sum(3 * n * 4 for n in C2_NS))

    def one_pass(lo: float = 0.0, hi: float = 1.0, stacked: bool = True):
        def cols(n):
            return int(n * lo), int(n * hi)
        a3, b3 = cols(S)
        rows3 = [c3[r, a3:b3] for r in range(C3_W)]
        if stacked:
            oracle.fold_stacked(c3)
        else:
            oracle.fold(rows3)  # a column range of a stack is not contiguous
        oracle.fold(rows3)
        a = [c4[r, a3:b3].copy() for r in range(C4_W)]
        oracle.allreduce(a, s4)
        a = [c4[r, a3:b3].copy() for r in range(C4_W)]
        oracle.staged_allreduce(a, s4)
        a5, b5 = cols(C5_N)
        for W in C5_WS:
            m = oracle.mean_scale(W)
            oracle.scale(oracle.fold([c5[W][r, a5:b5] for r in range(W)]), m)
            a = [c5[W][r, a5:b5].copy() for r in range(W)]
            oracle.allreduce(a, m)
        for n in C2_NS:
            a2, b2 = cols(n)
            if a2 < b2:
                oracle.fold([c2[n][r, a2:b2] for r in range(2)])

    t0 = time.perf_counter()
    passes = 0
    while True:
        one_pass()
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    value = passes * pass_bytes / el / 1e9

    from concurrent.futures import ThreadPoolExecutor
    T = os.cpu_count() or 1
    with ThreadPoolExecutor(max_workers=T) as ex:
        def split_pass():
            list(ex.map(lambda k: one_pass(k / T, (k + 1) / T, stacked=False), range(T)))
        split_pass()  # warm the pool
        t0 = time.perf_counter()
        split_passes = 0
        while True:
            split_pass()
            split_passes += 1
            el_split = time.perf_counter() - t0
            if el_split >= split_budget_s:
                break
    return {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{passes} passes over the first 2^21 elements of every C3/C4 rank row "
                      f"and the full C5/C2 rows (all rows of one step), {el:.1f} s, "
                      f"single-threaded serial fold",
            "cpu_model": cpu_model(),
            "threads_split": {"value": round(split_passes * pass_bytes / el_split / 1e9, 3), "unit": "GB/s",
                              "cores": T,
                              "sample": f"the same sample, {split_passes} passes in {el_split:.1f} s, "
                                        f"every row's elements split into {T} contiguous ranges, "
                                        f"one thread each"}}


def run_gpu(args) -> None:
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import detfold_inputs as gen
    import deterministic_fixed_order_gb300 as df

    wl = Workload(torch, df, gen, dev)
    rows = wl.rows()
    bytes_by_row = row_bytes()
    step_bytes = sum(bytes_by_row.values())
    stream = torch.cuda.current_stream()

    peaks_run = copy_peak_gbs(torch, df, dev)
    copy_gbs = peaks_run["d2d_copy_gbs"]

    steps_done = 0

    def do_step():
        nonlocal steps_done
        for _, fn, _ in rows:
            fn()
        steps_done += 1

    for _ in range(args.warmup):
        do_step()
    torch.cuda.synchronize()

    K = args.steps
    K_rows = min(K, 20)  # instrumented steps for the per-row times
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in rows] for _ in range(K_rows)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # untimed load so that every clock sample is taken with the GPU busy
        t_pre = time.perf_counter()
        while time.perf_counter() - t_pre < 1.0:
            do_step()
            torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        # the timed region: K whole steps, nothing recorded between rows (an
        # event between two launches would stop the second from overlapping
        # the first's tail)
        start.record(stream)
        for k in range(K):
            do_step()
        end.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        # per-row times from further steps with an event pair around each row
        for k in range(K_rows):
            for j, (_, fn, _) in enumerate(rows):
                ev[k][j][0].record(stream)
                fn()
                ev[k][j][1].record(stream)
            steps_done += 1
        torch.cuda.synchronize()
    clock_summary = clk.summary()
    ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    ms_per_step = ms / K
    value = whole_job_gbs(world, step_bytes, ms_per_step)

    per_row = {}
    launches = 0
    for j, (name, _, nl) in enumerate(rows):
        tms = [ev[k][j][0].elapsed_time(ev[k][j][1]) for k in range(K_rows)]
        avg = sum(tms) / K_rows
        per_row[name] = {"ms": round(avg, 5), "gbs": round(bytes_by_row[name] / (avg * 1e-3) / 1e9, 1)}
        launches += nl * K
    peak, peak_src = peaks()
    for name in per_row:
        per_row[name]["frac"] = round(per_row[name]["gbs"] / peak, 4)

    # dominant single-kernel rows: the W=8 fold kernel (c3_stacked + c3_ptrs
    # run the same instantiation) against the fused all-reduce kernel
    c3_ms = (per_row["c3_stacked"]["ms"] + per_row["c3_ptrs"]["ms"]) / 2
    c4_ms = per_row["c4_fused"]["ms"]
    if 2 * c3_ms >= c4_ms:
        dom, dom_bytes, dom_ms = ("fold_bulk_kernel<W=8,sum> (c3_stacked+c3_ptrs)",
                                  bytes_by_row["c3_stacked"], c3_ms)
    else:
        dom, dom_bytes, dom_ms = ("fold_bulk_kernel<W=4,all-reduce> (c4_fused)",
                                  bytes_by_row["c4_fused"], c4_ms)
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    khash = kernel_source_hash()
    tr = NCU_TRAFFIC.get(dom.split(" ")[0])
    traffic = tr["bytes_per_launch"] if tr and tr.get("kernel_hash") == khash else None
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "frac_note": "frac = achieved / peak, peak = the measured copy rate of MEASURED_PEAKS.json "
                             "(a torch device copy, not the HBM3e nominal); above 1 means the fold "
                             "streams faster than that copy; frac_of_nominal is against 7900 GB/s",
                "algorithmic_bytes_per_launch": dom_bytes,
                "frac_of_d2d_copy_this_run": round(achieved / peaks_run["d2d_copy_gbs"], 4),
                "frac_of_stream_kernel_this_run": round(achieved / peaks_run["stream_kernel_gbs"], 4),
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4)}

    rng = np.random.default_rng(1234)
    step_samples = collect_step_samples(wl, steps_done, rng)

    graph = graph_us_per_call(torch, df, wl)
    graph_samples = graph.pop("_specs")
    extra_rows = next_rows(torch, df, wl)
    c5_launch = c5_launches(torch, df, wl)

    # End to end through the public API with host buffers: every step copies
    # the step's inputs from pinned host memory, runs every row, and reads
    # back every result. Every input crosses the link once: a row that folds
    # in place an input another call also reads gets its copy on the device
    # (dup_rows). Three streams pipeline the rows: uploads run ahead on an
    # H2D stream, the calls run on the compute stream as each row's inputs
    # land, and results drain on a D2H stream, so the two link directions
    # overlap. Events keep a buffer from being overwritten before the previous
    # step has finished reading it.
    e2e_steps = max(3, min(20, K))
    pin = lambda n: torch.empty(n, dtype=torch.float32, pin_memory=True)
    h_out = {"c3": pin(C3_N), "c3b": pin(C3_N), "c4f": pin(C4_W * C4_N), "c4s": pin(C4_W * C4_N)}
    for W in C5_WS:
        h_out[f"c5s{W}"] = pin(C5_N)
        h_out[f"c5a{W}"] = pin(W * C5_N)
    for n in C2_NS:
        h_out[f"c2{n}"] = pin(n)
    def io_of(w):
        """(row name -> [(device dst, host src)], [(host dst, device src)]) of
        one set of device buffers."""
        io = {
            "c3_stacked": ([(w.c3, w.h_c3)], [(h_out["c3"], w.c3_out)]),
            "c3_ptrs": ([], [(h_out["c3b"], w.c3_out2)]),
            "c4_fused": ([(w.c4f[r], w.h_c4[r * C4_N:(r + 1) * C4_N]) for r in range(C4_W)],
                         [(h_out["c4f"][r * C4_N:(r + 1) * C4_N], w.c4f[r]) for r in range(C4_W)]),
            # the staged row folds the same C4 input as the fused row: it
            # crosses the link once (with the fused row) and is duplicated on
            # the device (dup_rows below)
            "c4_staged": ([], [(h_out["c4s"][r * C4_N:(r + 1) * C4_N], w.c4s[r]) for r in range(C4_W)]),
        }
        for W in C5_WS:
            # the sum's sources cross the link; the all-reduce's arenas, the
            # same rows, are copied from them on the device (dup_rows)
            ins, outs = [], [(h_out[f"c5s{W}"], w.c5_out[W])]
            for r in range(W):
                ins.append((w.c5_sum_src[W][r], w.h_c5[W][r * C5_N:(r + 1) * C5_N]))
                outs.append((h_out[f"c5a{W}"][r * C5_N:(r + 1) * C5_N], w.c5_ar[W][r]))
            io[f"c5_w{W}"] = (ins, outs)
        for n in C2_NS:
            io[f"c2_{n}"] = ([(w.c2[n], w.h_c2[n])], [(h_out[f"c2{n}"], w.c2_out[n])])
        return io

    # Two sets of device buffers, alternate steps: the uploads of step k+1
    # never wait for the read-back of step k (an in-place all-reduce's inputs
    # are its outputs), so the two directions of the host link overlap. Every
    # step still uploads all its inputs and reads back all its results.
    sets = [(wl, rows, io_of(wl))]
    twin = wl.device_twin()
    sets.append((twin, twin.rows(), io_of(twin)))
    io = sets[0][2]
    h2d = sum(d.numel() * 4 for ins, _ in io.values() for d, _ in ins)
    # every input crosses the link once per step, no more
    assert h2d == step_input_bytes(), (h2d, step_input_bytes())
    d2h = sum(h.numel() * 4 for _, outs in io.values() for h, _ in outs)
    # one upload and one download stream per row: a row whose buffers are
    # still being read back does not hold up the other rows' uploads
    s_h2d = {name: torch.cuda.Stream(device=dev) for name, _, _ in rows}
    s_d2h = {name: torch.cuda.Stream(device=dev) for name, _, _ in rows}
    s_cmp = torch.cuda.Stream(device=dev)
    ev_cmp = [{name: None for name, _, _ in rows} for _ in sets]
    ev_d2h = [{name: None for name, _, _ in rows} for _ in sets]
    # rows that also read a row's uploaded inputs (c3_ptrs folds the C3 rows)
    also_reads = {"c3_stacked": ["c3_ptrs"]}
    # inputs uploaded with one row and copied on the device, before that row
    # runs, into the buffers of a second row that folds them in place too:
    # row -> (receiving row, [(device dst, device src)] of a buffer set)
    dup_rows = {"c4_fused": ("c4_staged", lambda w: [(w.c4s[r], w.c4f[r]) for r in range(C4_W)])}
    for W in C5_WS:
        dup_rows[f"c5_w{W}"] = (f"c5_w{W}", lambda w, W=W: [(w.c5_ar[W][r], w.c5_sum_src[W][r]) for r in range(W)])
    dup_bytes = sum(2 * d.numel() * 4 for _, (_, pairs) in dup_rows.items() for d, _ in pairs(wl))
    step_no = [0]

    def e2e_step(compute: bool = True):
        k = step_no[0] % 2
        step_no[0] += 1
        set_w, set_rows, set_io = sets[k]
        for name, fn, _ in set_rows:
            ins, outs = set_io[name]
            up, down = s_h2d[name], s_d2h[name]
            with torch.cuda.stream(up):
                for ev in [ev_cmp[k][name], ev_d2h[k][name]] + [ev_cmp[k][x] for x in also_reads.get(name, [])]:
                    if ev is not None:
                        up.wait_event(ev)
                for d, h in ins:
                    d.copy_(h, non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(up)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(landed)
                if ev_d2h[k][name] is not None:
                    s_cmp.wait_event(ev_d2h[k][name])
                if compute and name in dup_rows:
                    dst_row, pairs = dup_rows[name]
                    if ev_d2h[k][dst_row] is not None:  # its last read-back is done
                        s_cmp.wait_event(ev_d2h[k][dst_row])
                    for d, src in pairs(set_w):
                        df.detfold_broadcast([d], 1, src, src.numel())
                if compute:
                    fn()
                ev_cmp[k][name] = torch.cuda.Event()
                ev_cmp[k][name].record(s_cmp)
            with torch.cuda.stream(down):
                down.wait_event(ev_cmp[k][name])
                for h, d in outs:
                    h.copy_(d, non_blocking=True)
                ev_d2h[k][name] = torch.cuda.Event()
                ev_d2h[k][name].record(down)

    for _ in range(4):  # both sets twice before timing: first copies from fresh pinned buffers run slow
        e2e_step()
    torch.cuda.synchronize()

    def e2e_pass(compute: bool = True) -> float:
        """ms per step over one pass of e2e_steps pipelined steps (without
        their kernels when compute is False: the link's time for the same
        transfers on the same schedule)."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(s_cmp)
        for st_ in list(s_h2d.values()) + list(s_d2h.values()):
            st_.wait_event(e0)
        for _ in range(e2e_steps):
            e2e_step(compute)
        for st_ in list(s_h2d.values()) + list(s_d2h.values()):
            done = torch.cuda.Event()
            done.record(st_)
            s_cmp.wait_event(done)
        e1.record(s_cmp)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)

    # the host link is measured before and after the passes, in this run,
    # and after each pass the same transfers run as a pass of their own with
    # no kernels: the end-to-end figure is link-bound, so it is read against
    # the link's own rate at the time

    link_before = host_link_gbs(torch, dev)
    sample = LinkSample(torch, dev)
    pass_ms, pass_link, pass_copies = [], [], []
    for _ in range(E2E_PASSES):
        pass_ms.append(e2e_pass())
        pass_copies.append(e2e_pass(compute=False))
        pass_link.append(sample())
    del sample
    e2e_step()  # leave the last results of a real step in the host buffers
    e2e_step()
    torch.cuda.synchronize()
    link = host_link_gbs(torch, dev)
    e2e_ms = statistics.median(pass_ms)
    e2e_value = whole_job_gbs(world, step_bytes, e2e_ms)
    link_gbs = (h2d + d2h) / (e2e_ms * 1e-3) / 1e9
    pass_gbs = sorted(whole_job_gbs(world, step_bytes, m) for m in pass_ms)
    # every step starts from the host inputs, so the read-back is one step
    idx = np.arange(0, C3_N, 16411)
    idx4 = np.arange(0, C4_N, 24593)
    h4 = wl.h_c4.numpy().reshape(C4_W, C4_N)
    e2e_samples = [
        {"group": "e2e", "kind": "fold_stacked",
         "inputs": np.ascontiguousarray(wl.h_c3.numpy().reshape(C3_W, C3_N)[:, idx]),
         "got": [h_out["c3"].numpy()[idx]]},
        {"group": "e2e", "kind": "allreduce", "repeat": 1, "scale": wl.scale4,
         "inputs": [np.ascontiguousarray(h4[r, idx4]) for r in range(C4_W)],
         "got": [[h_out["c4f"].numpy()[r * C4_N + idx4] for r in range(C4_W)],
                 [h_out["c4s"].numpy()[r * C4_N + idx4] for r in range(C4_W)]]},
    ]

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cpu, check = oracle_leg(gen, world, step_samples + graph_samples + e2e_samples)
    for n in C2_NS:
        graph[str(n)]["words_differing_after_replays"] = check.pop(f"c2_{n}_after_graph_replays")
    e2e_check = check.pop("e2e")
    check["words_differing"] = int(sum(check.values()))

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "us_per_call_16KiB_W2": graph["4096"]["us_per_call"],
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded xorshift64 generators: C1/C2 vecf, C3 gradient-like, "
                "C4 normal, C5 stress)",
        "config": arm_config(world),
        "value_note": "algorithmic bytes of the whole step over its device time: every row, including "
                      "the staged comparator (charged 2W len-units, moves 4W+1) and the latency-bound "
                      "small-payload rows; rows[*].frac and roofline are the per-kernel evidence",
        "rows": per_row,
        "roofline": roofline,
        "c2_graph": graph,
        "next_rows": extra_rows,
        "c5_launches": c5_launch,
        "copy_peak_gbs_this_run": round(copy_gbs, 1),
        "peaks_this_run": {"d2d_copy_gbs": round(peaks_run["d2d_copy_gbs"], 1),
                           "stream_kernel_gbs": round(peaks_run["stream_kernel_gbs"], 1),
                           "nominal_gbs": NOMINAL_HBM_GBS,
                           "method": "best of 20, 1 GiB read + 1 GiB written per call"},
        "bitwise_sampled": check,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "pipelined": "per-row H2D and D2H streams around one compute stream; two sets of "
                             "device buffers, alternate steps",
                "device_copies_per_step": dup_bytes,
                "device_copies_note": "every input crosses the link once: the staged C4 row's and the "
                                      "C5 all-reduces' in-place copies of inputs another call also "
                                      "folds are made on the device (detfold_broadcast), inside the "
                                      "timed region",
                "bitwise_sampled_words_differing": int(e2e_check),
                "link_bytes_gbs": round(link_gbs, 1),
                "passes": {"count": E2E_PASSES, "steps_each": e2e_steps,
                           "gbs_min": round(pass_gbs[0], 1), "gbs_median": round(e2e_value, 1),
                           "gbs_max": round(pass_gbs[-1], 1),
                           "each": [{"gbs": round(whole_job_gbs(world, step_bytes, m), 1),
                                     "ms_per_step": round(m, 2),
                                     "copies_only_ms_per_step": round(c, 2),
                                     "copies_only_of_e2e": round(c / m, 3),
                                     "link_step_gbs": round((h2d + d2h) / (m * 1e-3) / 1e9, 1),
                                     "link_sample_both_gbs": round(l, 1)}
                                    for m, c, l in zip(pass_ms, pass_copies, pass_link)]},
                "link_this_run": {k: round(v, 1) for k, v in link.items()},
                "link_before_passes": {k: round(v, 1) for k, v in link_before.items()},
                "link_utilisation_of_both_ways": round(link_gbs / link["both_gbs"], 3)},
        "gpu_launches": launches,
        "clocks": clock_summary,
        "cpu_baseline": cpu,
        "kernel_source_hash": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm (CPU oracle)

def run_reference(args) -> None:
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import detfold_inputs as gen
    import oracle
    # Each step: every row of the step on a bounded sample (the first S
    # elements of each rank's arena for the large rows, the full C5/C2 rows).
    S = 1 << 20
    c3 = gen.gradient_rows(C3_W, S)
    c4 = gen.normal_rows(C4_W, S)
    c5 = {W: gen.stress_rows(W, C5_N) for W in C5_WS}
    c2 = {n: gen.c1_rows(2, n) for n in C2_NS}
    s4 = np.float32(0.25)
    step_bytes = (2 * (C3_W + 1) * S * 4 + 2 * (2 * C4_W * S * 4)
                  + sum(((W + 1) + 2 + 2 * W) * C5_N * 4 for W in C5_WS)
                  + sum(3 * n * 4 for n in C2_NS))

    def step():
        oracle.fold_stacked(c3)
        oracle.fold(c3)
        a = [c4[r].copy() for r in range(C4_W)]
        oracle.allreduce(a, s4)
        a = [c4[r].copy() for r in range(C4_W)]
        oracle.staged_allreduce(a, s4)
        for W in C5_WS:
            m = oracle.mean_scale(W)
            oracle.scale(oracle.fold(c5[W]), m)
            a = [c5[W][r].copy() for r in range(W)]
            oracle.allreduce(a, m)
        for n in C2_NS:
            oracle.fold_stacked(c2[n])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = step_bytes / (ms * 1e-3) / 1e9
    sample = ("every row of the step on the first 2^20 elements of each C3/C4 rank row "
              "and the full C5/C2 rows; single-threaded serial oracle")
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": arm_config(world),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample,
                         "sample_step_algorithmic_bytes": step_bytes, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
