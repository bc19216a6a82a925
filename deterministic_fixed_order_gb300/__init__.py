"""Python binding of libdetfold, the fixed-order elementwise fold for GB300.

Argument marshalling only: every step of the fold runs in the CUDA library
(``libdetfold.so``, built in-tree from ``csrc/`` by ``build.build()``). If
the library has not been built this module raises on import; there is no
CPU fallback.

The functions keep the C names of ``include/detfold.h``. Device operands may
be given as CUDA float32 tensors (checked for device, dtype, contiguity and
size against the lengths passed) or as raw integer addresses (passed through
unchecked). ``stream`` may be None (torch's current stream), a
``torch.cuda.Stream`` or a raw handle. A negative status raises
``DetfoldError``; the ``status_*`` variants return it instead.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = [
    "DetfoldError", "lib", "DETFOLD_MAX_W", "DETFOLD_MAX_LEN",
    "DETFOLD_STAGED_REVERSE_DELIVERY", "DETFOLD_STAGED_SEPARATE_SCALE", "DETFOLD_STAGED_CE_COPIES",
    "detfold_broadcast", "detfold_all_gather", "detfold_sum_ptrs_dev",
    "detfold_loopback_allreduce_dev", "device_table", "detfold_one_shot_allreduce", "OneShotLink",
    "detfold_sum_stacked", "detfold_sum_ptrs", "detfold_scale",
    "detfold_loopback_allreduce", "detfold_mean_scale", "detfold_staged_workspace_bytes",
    "detfold_loopback_allreduce_staged", "detfold_loopback_allreduce_staged_ex",
    "detfold_loopback_allreduce_staged_noalloc", "detfold_shard_plan", "detfold_status_string",
    "detfold_last_cuda_error", "detfold_pipeline_timeouts", "STATUS",
]

LIB_PATH = _build.LIB

DETFOLD_MAX_W = 256
DETFOLD_MAX_LEN = 1 << 40
DETFOLD_STAGED_REVERSE_DELIVERY = 1
DETFOLD_STAGED_SEPARATE_SCALE = 2
DETFOLD_STAGED_CE_COPIES = 4

STATUS = {
    "DETFOLD_OK": 0, "DETFOLD_ERR_NULL": -1, "DETFOLD_ERR_WORLD": -2, "DETFOLD_ERR_LEN": -3,
    "DETFOLD_ERR_ALIGN": -4, "DETFOLD_ERR_OVERLAP": -5, "DETFOLD_ERR_WORKSPACE": -6,
    "DETFOLD_ERR_CUDA": -7, "DETFOLD_ERR_ARG": -8, "DETFOLD_ERR_SCRATCH_LIMIT": -9,
}
DETFOLD_NOALLOC_SCRATCH_BYTES = 16 << 20
DETFOLD_ONESHOT_MAX_W = 64
DETFOLD_ONESHOT_MAX_LEN = 1 << 22
DETFOLD_ONESHOT_MAX_CTAS = 1024
DETFOLD_ONESHOT_LINK_BYTES = 2 * DETFOLD_ONESHOT_MAX_CTAS * 8 + 64
DETFOLD_ONESHOT_REFUSE_ENTRY = 40043
DETFOLD_ONESHOT_REFUSE_EXIT = 40044

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libdetfold.so is not built ({LIB_PATH}); run "
        "`python -c 'import __graft_entry__ as g; g.build()'` first")

lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_F = ctypes.c_float

lib.detfold_sum_stacked.argtypes = [_P, _P, _INT, _I64, _P]
lib.detfold_sum_ptrs.argtypes = [_P, _P, _INT, _I64, _P]
lib.detfold_scale.argtypes = [_P, _I64, _F, _P]
lib.detfold_loopback_allreduce.argtypes = [_P, _INT, _I64, _F, _P]
lib.detfold_staged_workspace_bytes.argtypes = [_I64, _INT]
lib.detfold_staged_workspace_bytes.restype = _I64
lib.detfold_mean_scale.argtypes = [_INT, _P]
lib.detfold_loopback_allreduce_staged.argtypes = [_P, _INT, _I64, _F, _P, _I64, _P]
lib.detfold_loopback_allreduce_staged_ex.argtypes = [_P, _INT, _I64, _F, _INT, _P, _I64, _P]
lib.detfold_loopback_allreduce_staged_noalloc.argtypes = [_P, _INT, _I64, _F, _INT, _P]
lib.detfold_broadcast.argtypes = [_P, _INT, _P, _I64, _P]
lib.detfold_sum_ptrs_dev.argtypes = [_P, _P, _INT, _I64, _P, _P]
lib.detfold_one_shot_allreduce.argtypes = [_P, _INT, _I64, _F, _P, ctypes.c_uint64, _P, _P, _I64,
                                           _INT, _INT, _P]
lib.detfold_loopback_allreduce_dev.argtypes = [_P, _INT, _I64, _F, _P, _P]
lib.detfold_all_gather.argtypes = [_P, _INT, _P, _I64, _P]
lib.detfold_shard_plan.argtypes = [_I64, _INT, _P, _P]
lib.detfold_status_string.argtypes = [_INT]
lib.detfold_status_string.restype = ctypes.c_char_p
lib.detfold_last_cuda_error.argtypes = []
lib.detfold_pipeline_timeouts.argtypes = [_P]
for _name in ("detfold_sum_stacked", "detfold_sum_ptrs", "detfold_scale",
              "detfold_loopback_allreduce", "detfold_mean_scale", "detfold_loopback_allreduce_staged",
              "detfold_loopback_allreduce_staged_ex", "detfold_loopback_allreduce_staged_noalloc",
              "detfold_broadcast", "detfold_sum_ptrs_dev", "detfold_loopback_allreduce_dev",
              "detfold_one_shot_allreduce", "detfold_all_gather", "detfold_shard_plan",
              "detfold_last_cuda_error", "detfold_pipeline_timeouts"):
    getattr(lib, _name).restype = _INT


class DetfoldError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib.detfold_status_string(status).decode()
        if status == STATUS["DETFOLD_ERR_CUDA"]:
            msg += f" (cudaError {lib.detfold_last_cuda_error()})"
        super().__init__(f"{where}: status {status}: {msg}")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != 0:
        raise DetfoldError(status, where)


_torch = None          # torch, imported on first use
_F32 = None
_cuda_ok = None        # torch.cuda.is_available(), asked once
_raw_stream = None     # torch's raw current-stream query, if this torch has it
_ARRAYS = {}           # ctypes pointer-array types by length


def _t():
    global _torch, _F32
    if _torch is None:
        import torch
        _torch, _F32 = torch, torch.float32
    return _torch


def _label(what: str, k) -> str:
    return what if k is None else f"{what}[{k}]"


def _dev_ptr(x, need_elems: int | None, what: str, k=None) -> int:
    """Address of a device operand; tensors are checked against need_elems.
    (The checks run on every call; the messages are built only on failure.)"""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    torch = _torch or _t()
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{_label(what, k)}: expected a CUDA float32 tensor or an int address")
    if not x.is_cuda or x.dtype is not _F32:
        raise TypeError(f"{_label(what, k)}: expected a CUDA float32 tensor, got {x.device} {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{_label(what, k)}: tensor must be contiguous")
    if need_elems is not None and x.numel() < need_elems:
        raise ValueError(f"{_label(what, k)}: tensor holds {x.numel()} elements, call needs {need_elems}")
    return x.data_ptr()


def _current_stream() -> int:
    """Handle of torch's current stream on the current device (0 without CUDA).
    After the first call initializes torch's CUDA state through the public
    API, the handle comes from torch's raw stream query, which skips building
    a Stream object."""
    global _cuda_ok, _raw_stream
    if _cuda_ok is None:
        torch = _t()
        _cuda_ok = torch.cuda.is_available()
        if _cuda_ok:
            torch.cuda.init()
            _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if not _cuda_ok:
        return 0
    if _raw_stream is not None:
        return _raw_stream(_torch._C._cuda_getDevice())
    return _torch.cuda.current_stream().cuda_stream


def _stream(s) -> int:
    if s is None:
        return _current_stream()
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ptr_array(items, need_elems, what):
    ptrs = [_dev_ptr(t, need_elems, what, k) for k, t in enumerate(items)]
    n = max(1, len(ptrs))
    arr = _ARRAYS.get(n)
    if arr is None:
        arr = _ARRAYS.setdefault(n, ctypes.c_void_p * n)
    return arr(*ptrs)


# ------------------------------------------------------------------ status-returning calls

def status_sum_stacked(out, stacked, W: int, length: int, stream=None) -> int:
    return lib.detfold_sum_stacked(_dev_ptr(out, length, "out"),
                                   _dev_ptr(stacked, W * length, "stacked"),
                                   W, length, _stream(stream))


def status_sum_ptrs(out, srcs, W: int, length: int, stream=None) -> int:
    tab = _ptr_array(srcs, length, "srcs") if srcs is not None else None
    return lib.detfold_sum_ptrs(_dev_ptr(out, length, "out"), tab, W, length, _stream(stream))


def status_scale(buf, length: int, scale: float, stream=None) -> int:
    return lib.detfold_scale(_dev_ptr(buf, length, "buf"), length, scale, _stream(stream))


def status_loopback_allreduce(arenas, W: int, length: int, mean_scale: float = 1.0,
                              stream=None) -> int:
    tab = _ptr_array(arenas, length, "arenas") if arenas is not None else None
    return lib.detfold_loopback_allreduce(tab, W, length, mean_scale, _stream(stream))


def _workspace_ptr(ws, workspace_bytes: int) -> int:
    if ws is None or isinstance(ws, int):
        return ws or 0
    if not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace: expected a contiguous CUDA tensor")
    if ws.numel() * ws.element_size() < workspace_bytes:
        raise ValueError("workspace: tensor smaller than workspace_bytes")
    return ws.data_ptr()


def status_loopback_allreduce_staged(arenas, W: int, length: int, mean_scale: float, workspace,
                                     workspace_bytes: int, stream=None) -> int:
    tab = _ptr_array(arenas, length, "arenas") if arenas is not None else None
    return lib.detfold_loopback_allreduce_staged(tab, W, length, mean_scale,
                                                 _workspace_ptr(workspace, workspace_bytes),
                                                 workspace_bytes, _stream(stream))


def status_loopback_allreduce_staged_ex(arenas, W: int, length: int, mean_scale: float, flags: int,
                                        workspace, workspace_bytes: int, stream=None) -> int:
    tab = _ptr_array(arenas, length, "arenas") if arenas is not None else None
    return lib.detfold_loopback_allreduce_staged_ex(tab, W, length, mean_scale, flags,
                                                    _workspace_ptr(workspace, workspace_bytes),
                                                    workspace_bytes, _stream(stream))


def status_loopback_allreduce_staged_noalloc(arenas, W: int, length: int, mean_scale: float,
                                             flags: int, stream=None) -> int:
    tab = _ptr_array(arenas, length, "arenas") if arenas is not None else None
    return lib.detfold_loopback_allreduce_staged_noalloc(tab, W, length, mean_scale, flags,
                                                         _stream(stream))


def status_broadcast(dsts, ndst: int, src, length: int, stream=None) -> int:
    tab = _ptr_array(dsts, length, "dsts") if dsts is not None else None
    return lib.detfold_broadcast(tab, ndst, _dev_ptr(src, length, "src"), length, _stream(stream))


def status_all_gather(outs, W: int, parts, span: int, stream=None) -> int:
    otab = _ptr_array(outs, W * span, "outs") if outs is not None else None
    ptab = _ptr_array(parts, span, "parts") if parts is not None else None
    return lib.detfold_all_gather(otab, W, ptab, span, _stream(stream))


def _table_ptr(table, W: int) -> int:
    """Address of a device pointer table: a CUDA int64 tensor of >= W entries, or an int."""
    if isinstance(table, int):
        return table
    torch = _torch or _t()
    if not isinstance(table, torch.Tensor) or not table.is_cuda or table.dtype != torch.int64:
        raise TypeError("table: expected a CUDA int64 tensor of device addresses")
    if not table.is_contiguous() or table.numel() < W:
        raise ValueError(f"table: needs {W} contiguous entries, has {table.numel()}")
    return table.data_ptr()


def _status_ptr(status) -> int:
    if status is None or isinstance(status, int):
        return status or 0
    torch = _torch or _t()
    if not status.is_cuda or status.dtype != torch.int32 or status.numel() < 1:
        raise TypeError("status: expected a CUDA int32 tensor")
    return status.data_ptr()


def device_table(tensors, device=None):
    """A CUDA int64 tensor holding the data addresses of `tensors` (for the
    *_dev entry points). Each tensor must be a CUDA float32 tensor."""
    torch = _torch or _t()
    ptrs = [_dev_ptr(t, None, f"tensors[{k}]") for k, t in enumerate(tensors)]
    dev = device if device is not None else tensors[0].device
    return torch.tensor(ptrs, dtype=torch.int64, device=dev)


def status_sum_ptrs_dev(out, table, W: int, length: int, status=None, stream=None) -> int:
    return lib.detfold_sum_ptrs_dev(_dev_ptr(out, length, "out"), _table_ptr(table, W), W, length,
                                    _status_ptr(status), _stream(stream))


def status_loopback_allreduce_dev(table, W: int, length: int, mean_scale: float = 1.0,
                                  status=None, stream=None) -> int:
    return lib.detfold_loopback_allreduce_dev(_table_ptr(table, W), W, length, mean_scale,
                                              _status_ptr(status), _stream(stream))


def _raw_dev(x, nbytes: int, what: str) -> int:
    """Address of a CUDA tensor of at least nbytes (any dtype), or an int."""
    if isinstance(x, int):
        return x
    torch = _torch or _t()
    if not isinstance(x, torch.Tensor) or not x.is_cuda or not x.is_contiguous():
        raise TypeError(f"{what}: expected a contiguous CUDA tensor")
    if x.numel() * x.element_size() < nbytes:
        raise ValueError(f"{what}: needs {nbytes} bytes, has {x.numel() * x.element_size()}")
    return x.data_ptr()


def status_one_shot_allreduce(arenas, W: int, length: int, mean_scale: float, link, epoch: int,
                              stage, words, wait_ns: int = 1_000_000_000, drop_rank: int = -1,
                              drop_at_exit: int = 0, stream=None) -> int:
    tab = _ptr_array(arenas, length, "arenas") if arenas is not None else None
    return lib.detfold_one_shot_allreduce(
        tab, W, length, mean_scale, _raw_dev(link, DETFOLD_ONESHOT_LINK_BYTES, "link"), epoch,
        _raw_dev(stage, W * length * 4, "stage"), _raw_dev(words, W * 4, "words"), wait_ns,
        drop_rank, drop_at_exit, _stream(stream))


# ------------------------------------------------------------------ raising calls (C names)

def detfold_sum_stacked(out, stacked, W: int, length: int, stream=None) -> None:
    _check(status_sum_stacked(out, stacked, W, length, stream), "detfold_sum_stacked")


def detfold_sum_ptrs(out, srcs, W: int, length: int, stream=None) -> None:
    _check(status_sum_ptrs(out, srcs, W, length, stream), "detfold_sum_ptrs")


def detfold_scale(buf, length: int, scale: float, stream=None) -> None:
    _check(status_scale(buf, length, scale, stream), "detfold_scale")


def detfold_loopback_allreduce(arenas, W: int, length: int, mean_scale: float = 1.0,
                               stream=None) -> None:
    _check(status_loopback_allreduce(arenas, W, length, mean_scale, stream),
           "detfold_loopback_allreduce")


def detfold_staged_workspace_bytes(length: int, W: int) -> int:
    n = lib.detfold_staged_workspace_bytes(length, W)
    _check(n if n < 0 else 0, "detfold_staged_workspace_bytes")
    return n


def detfold_mean_scale(W: int) -> float:
    """fl(1/W) in binary32, computed by the library: the mean's multiplier."""
    out = ctypes.c_float(0.0)
    _check(lib.detfold_mean_scale(W, ctypes.byref(out)), "detfold_mean_scale")
    return out.value


def detfold_loopback_allreduce_staged(arenas, W: int, length: int, mean_scale: float = 1.0,
                                      workspace=None, workspace_bytes: int = 0,
                                      stream=None) -> None:
    _check(status_loopback_allreduce_staged(arenas, W, length, mean_scale, workspace,
                                            workspace_bytes, stream),
           "detfold_loopback_allreduce_staged")


def detfold_loopback_allreduce_staged_ex(arenas, W: int, length: int, mean_scale: float = 1.0,
                                         flags: int = 0, workspace=None, workspace_bytes: int = 0,
                                         stream=None) -> None:
    """The staged all-reduce with the comparator's variants (DETFOLD_STAGED_*
    flags: reverse delivery, a separate mean pass, copy-engine copies)."""
    _check(status_loopback_allreduce_staged_ex(arenas, W, length, mean_scale, flags, workspace,
                                               workspace_bytes, stream),
           "detfold_loopback_allreduce_staged_ex")


def detfold_loopback_allreduce_staged_noalloc(arenas, W: int, length: int,
                                              mean_scale: float = 1.0, flags: int = 0,
                                              stream=None) -> None:
    """The staged all-reduce with its scratch inside the library (no device
    allocation by anyone): for callers that cannot allocate, such as code
    running during CUDA-graph capture or under a fixed device-memory budget.
    Requests larger than DETFOLD_NOALLOC_SCRATCH_BYTES of workspace raise
    DETFOLD_ERR_SCRATCH_LIMIT; concurrent calls on unordered streams race on
    the shared scratch."""
    _check(status_loopback_allreduce_staged_noalloc(arenas, W, length, mean_scale, flags, stream),
           "detfold_loopback_allreduce_staged_noalloc")


def detfold_sum_ptrs_dev(out, table, W: int, length: int, status=None, stream=None) -> None:
    """Fold over a device-resident pointer table (see include/detfold.h).
    The table's entries are not visible to the host: they must address
    `length` floats each, as the caller guarantees."""
    _check(status_sum_ptrs_dev(out, table, W, length, status, stream), "detfold_sum_ptrs_dev")


def detfold_loopback_allreduce_dev(table, W: int, length: int, mean_scale: float = 1.0,
                                   status=None, stream=None) -> None:
    _check(status_loopback_allreduce_dev(table, W, length, mean_scale, status, stream),
           "detfold_loopback_allreduce_dev")


def detfold_one_shot_allreduce(arenas, W: int, length: int, mean_scale: float, link, epoch: int,
                               stage, words, wait_ns: int = 1_000_000_000, drop_rank: int = -1,
                               drop_at_exit: int = 0, stream=None) -> None:
    _check(status_one_shot_allreduce(arenas, W, length, mean_scale, link, epoch, stage, words,
                                     wait_ns, drop_rank, drop_at_exit, stream),
           "detfold_one_shot_allreduce")


class OneShotLink:
    """Device state of one emulated one-shot link between W ranks: barrier
    flags and an epoch counter (zero-filled once), W stage rows of up to
    max_len floats, and the W refusal words."""

    def __init__(self, W: int, max_len: int, device="cuda"):
        torch = _torch or _t()
        self.W, self.max_len = W, max_len
        self.link = torch.zeros(DETFOLD_ONESHOT_LINK_BYTES // 8, dtype=torch.int64, device=device)
        self.stage = torch.empty(max(1, W * max_len), dtype=torch.float32, device=device)
        self.words = torch.zeros(W, dtype=torch.int32, device=device)

    def all_reduce(self, arenas, mean_scale: float = 1.0, wait_ns: int = 1_000_000_000,
                   drop_rank: int = -1, drop_at_exit: bool = False, stream=None,
                   epoch: int = 0) -> None:
        """One call. epoch 0 (the default): the link's device counter supplies
        the epoch, so the call can be captured in a CUDA graph and replayed;
        else the caller's epoch, larger than every epoch used on this link."""
        n = arenas[0].numel()
        if n > self.max_len or len(arenas) != self.W:
            raise ValueError("arenas do not fit this link")
        detfold_one_shot_allreduce(list(arenas), self.W, n, mean_scale, self.link, epoch,
                                   self.stage, self.words, wait_ns, drop_rank,
                                   1 if drop_at_exit else 0, stream)

    def counter(self) -> int:
        """The largest epoch used on this link so far (reads the device)."""
        return int(self.link[2 * DETFOLD_ONESHOT_MAX_CTAS].item())

    def barrier_errors(self) -> list[int]:
        """The refusal words of the last call: 0, 40043 (entry) or 40044 (exit)."""
        return [int(x) for x in self.words.cpu()]


def detfold_broadcast(dsts, ndst: int, src, length: int, stream=None) -> None:
    _check(status_broadcast(dsts, ndst, src, length, stream), "detfold_broadcast")


def detfold_all_gather(outs, W: int, parts, span: int, stream=None) -> None:
    _check(status_all_gather(outs, W, parts, span, stream), "detfold_all_gather")


def detfold_shard_plan(length: int, W: int) -> tuple[list[int], list[int]]:
    starts = (ctypes.c_int64 * max(1, W))()
    lens = (ctypes.c_int64 * max(1, W))()
    _check(lib.detfold_shard_plan(length, W, starts, lens), "detfold_shard_plan")
    return list(starts)[:W], list(lens)[:W]


def detfold_status_string(status: int) -> str:
    return lib.detfold_status_string(status).decode()


def detfold_last_cuda_error() -> int:
    return lib.detfold_last_cuda_error()


def detfold_pipeline_timeouts() -> int:
    """Bounded waits that ran out in the bulk-async path (should be 0).
    Synchronizes the device."""
    c = ctypes.c_int64(0)
    _check(lib.detfold_pipeline_timeouts(ctypes.byref(c)), "detfold_pipeline_timeouts")
    return c.value


# ------------------------------------------------------------------ tensor conveniences

def sum_stacked(stacked, out=None, stream=None):
    """out = fold of the rows of a [W, len] CUDA float32 tensor."""
    torch = _torch or _t()
    W, n = stacked.shape
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=stacked.device)
    detfold_sum_stacked(out, stacked, W, n, stream)
    return out


def sum_ptrs(srcs, out=None, stream=None):
    torch = _torch or _t()
    n = srcs[0].numel()
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=srcs[0].device)
    detfold_sum_ptrs(out, list(srcs), len(srcs), n, stream)
    return out


def loopback_allreduce(arenas, mean: bool = False, stream=None) -> None:
    W = len(arenas)
    scale = detfold_mean_scale(W) if mean else 1.0
    detfold_loopback_allreduce(list(arenas), W, arenas[0].numel(), scale, stream)


def mean_scale(W: int) -> float:
    """fl(1/W) in binary32, the scale the mean multiplies by (from the library)."""
    return detfold_mean_scale(W)


def shard_plan(length: int, W: int):
    return detfold_shard_plan(length, W)
