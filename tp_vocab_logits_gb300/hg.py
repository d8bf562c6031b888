"""Python binding of libhg (include/hg.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
computation of its own: it checks torch tensors' device, dtype, shape and
contiguity, turns them into raw device pointers, and calls the library. The
gather itself runs only in the library's CUDA kernels; if libhg.so cannot be
loaded every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

from . import _build

HG_OK, HG_ERR_ARG, HG_ERR_ROWS, HG_ERR_CAPTURE, HG_ERR_CUDA, HG_ERR_TIMEOUT, HG_ERR_STATE = range(7)
HG_MAX_TP = 32


class HGError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} (status {status})")


class _Options(ctypes.Structure):
    _fields_ = [("poll_timeout_ns", ctypes.c_uint64), ("elems_per_lane", ctypes.c_int),
                ("ctas", ctypes.c_int), ("prefetch", ctypes.c_int), ("cooperative", ctypes.c_int),
                ("device_parity", ctypes.c_int), ("autotune", ctypes.c_int),
                ("timeline_calls", ctypes.c_int)]


_LIB: ctypes.CDLL | None = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libhg.so (built in-tree by ``_build.build()``); raises if absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with tp_vocab_logits_gb300._build.build()")
    lib = ctypes.CDLL(path)
    vp, vpp, i, st = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_void_p
    lib.hg_create.argtypes = [i, i, i, ctypes.POINTER(i), i, ctypes.POINTER(vp)]
    lib.hg_create_ex.argtypes = [i, i, i, ctypes.POINTER(i), i, ctypes.POINTER(_Options),
                                 ctypes.POINTER(vp)]
    lib.hg_destroy.argtypes = [vp]
    lib.hg_gather.argtypes = [vp, vpp, vpp, i, st]
    lib.hg_gather_host.argtypes = [vp, vpp, vpp, i, st]
    lib.hg_sync.argtypes = [vp, st]
    lib.hg_rearm.argtypes = [vp, st]
    lib.hg_parity.argtypes = [vp]
    lib.hg_mailbox.argtypes = [vp, i, ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)]
    ip = ctypes.POINTER(i)
    lib.hg_launch_shape.argtypes = [vp, i, ip, ip, ip, ip]
    lib.hg_debug_skip_push.argtypes = [vp, i]
    lib.hg_stock_gather.argtypes = [i, i, vpp, vpp, i, st]
    lib.hg_gather_fused.argtypes = [vp, vpp, vpp, vpp, vpp, i, i, st]
    lib.hg_gather_stats.argtypes = [vp, vpp, vpp, i, vp, st]
    lib.hg_timeline.argtypes = [vp, ctypes.POINTER(vp), ip, ip, ip]
    lib.hg_probe.argtypes = [i, i, i, vp, st]
    lib.hg_probe_scratch_bytes.argtypes = [i, i]
    lib.hg_probe_scratch_bytes.restype = ctypes.c_size_t
    lib.hg_strerror.argtypes = [i]
    lib.hg_strerror.restype = ctypes.c_char_p
    for name in ("hg_create", "hg_create_ex", "hg_destroy", "hg_gather", "hg_gather_host",
                 "hg_sync", "hg_rearm",
                 "hg_parity", "hg_mailbox", "hg_launch_shape", "hg_debug_skip_push",
                 "hg_stock_gather", "hg_gather_fused", "hg_gather_stats", "hg_timeline",
                 "hg_probe"):
        getattr(lib, name).restype = i
    _LIB = lib
    return lib


def strerror(status: int) -> str:
    try:
        return load().hg_strerror(status).decode()
    except RuntimeError:
        return f"status {status}"


def _check(status: int, where: str) -> None:
    if status != HG_OK:
        raise HGError(status, where)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr_array(tensors: Sequence[torch.Tensor]):
    return (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


class Handle:
    """Owner of one hg_handle; freed by hg_destroy on close() or collection."""

    def __init__(self, ptr: int, tp: int, shard_cols: int, cap: int, rows):
        self.ptr = ptr
        self.tp, self.shard_cols, self.cap = tp, shard_cols, cap
        self.rows = frozenset(rows) if rows else frozenset(range(1, cap + 1))

    @property
    def V(self) -> int:
        return self.tp * self.shard_cols

    def close(self) -> None:
        if self.ptr:
            _check(load().hg_destroy(self.ptr), "hg_destroy")
            self.ptr = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def hg_create(tp: int, shard_cols: int, cap: int, rows: Sequence[int] | None = None, *,
              poll_timeout_ns: int = 0, elems_per_lane: int = 0, ctas: int = 0,
              prefetch: int = 0, cooperative: bool = False,
              device_parity: bool = False, autotune: bool = False,
              timeline_calls: int = 0) -> Handle:
    lib = load()
    rows = list(rows or [])
    arr = (ctypes.c_int * max(1, len(rows)))(*rows)
    out = ctypes.c_void_p()
    if poll_timeout_ns or elems_per_lane or ctas or prefetch or cooperative or device_parity \
            or autotune or timeline_calls:
        opt = _Options(poll_timeout_ns, elems_per_lane, ctas, prefetch, int(bool(cooperative)),
                       int(bool(device_parity)), int(bool(autotune)), int(timeline_calls))
        st = lib.hg_create_ex(tp, shard_cols, cap, arr, len(rows), ctypes.byref(opt),
                              ctypes.byref(out))
    else:
        st = lib.hg_create(tp, shard_cols, cap, arr, len(rows), ctypes.byref(out))
    _check(st, "hg_create")
    return Handle(out.value, tp, shard_cols, cap, rows)


def hg_destroy(h: Handle) -> None:
    h.close()


def _check_tensors(ts: Sequence[torch.Tensor], n: int, cols: int, M: int, what: str,
                   host: bool = False) -> None:
    if len(ts) != n:
        raise ValueError(f"{what}: expected {n} tensors, got {len(ts)}")
    for t in ts:
        if host:
            if not t.is_cuda and not t.is_pinned():
                raise ValueError(f"{what}: host tensors must be in page-locked memory")
        elif not t.is_cuda:
            raise ValueError(f"{what}: tensors must be on a CUDA device")
        if t.dtype not in (torch.bfloat16, torch.int16):
            raise ValueError(f"{what}: dtype must be bfloat16 (or its int16 bits), got {t.dtype}")
        if tuple(t.shape) != (M, cols) or not t.is_contiguous():
            raise ValueError(f"{what}: need contiguous [{M}, {cols}], got {tuple(t.shape)}")


def GatherCall(h: Handle, shards: Sequence[torch.Tensor], outs: Sequence[torch.Tensor], M: int,
               stream=None):
    """Marshalled arguments of one hg_gather call, reusable across calls with
    the same buffers: returns a callable that makes the call (raising HGError
    on a failed status). The callable is a small CPython object (the _hgcall
    extension) that calls the C entry point directly, so per-call host work
    is the C call itself. When any tensor is in (page-locked) host memory the
    call is hg_gather_host: the kernel reads and writes host memory directly
    over the host-device link."""
    host = any(not t.is_cuda for t in list(shards) + list(outs))
    _check_tensors(shards, h.tp, h.shard_cols, M, "shards", host)
    _check_tensors(outs, h.tp, h.V, M, "outs", host)
    entry = load().hg_gather_host if host else load().hg_gather
    fn = ctypes.cast(entry, ctypes.c_void_p).value
    return _pycall().Call(fn, h, [t.data_ptr() for t in shards], [t.data_ptr() for t in outs],
                          M, _stream_ptr(stream), (list(shards), list(outs)), _raise_gather)


def _raise_gather(status: int) -> None:
    raise HGError(status, "hg_gather")


_PYCALL = None


def _pycall():
    """The _hgcall extension (built in-tree next to libhg.so); raises if absent."""
    global _PYCALL
    if _PYCALL is None:
        import importlib
        if not os.path.exists(_build.PYCALL):
            raise RuntimeError(f"{_build.PYCALL} is missing: build it with "
                               "tp_vocab_logits_gb300._build.build()")
        _PYCALL = importlib.import_module("tp_vocab_logits_gb300._hgcall")
    return _PYCALL


def hg_gather(h: Handle, shards: Sequence[torch.Tensor], outs: Sequence[torch.Tensor],
              M: int | None = None, stream=None) -> None:
    """One gather: shards[r] is rank r's [M, W] bf16 logits, outs[d] rank d's
    [M, V] bf16 output (both lists of device tensors)."""
    M = shards[0].shape[0] if M is None else M
    GatherCall(h, shards, outs, M, stream)()


def hg_gather_host(h: Handle, shards: Sequence[torch.Tensor], outs: Sequence[torch.Tensor],
                   M: int | None = None, stream=None) -> None:
    """One gather whose shards and outputs are page-locked host tensors
    (``tensor.pin_memory()``) or device tensors: the kernel reads and writes
    host memory directly."""
    M = shards[0].shape[0] if M is None else M
    GatherCall(h, shards, outs, M, stream)()


def hg_gather_fused(h: Handle, hidden: Sequence[torch.Tensor], weight: Sequence[torch.Tensor],
                    outs: Sequence[torch.Tensor], M: int | None = None,
                    logits: Sequence[torch.Tensor] | None = None, stream=None) -> None:
    """LM head + gather in one launch: hidden[r] is rank r's [M, K] bf16 input,
    weight[r] its [W, K] bf16 lm_head weight (nn.Linear layout), outs[d] rank
    d's [M, V] output; logits, if given, receives each rank's [M, W] bf16
    logits."""
    M = hidden[0].shape[0] if M is None else M
    K = hidden[0].shape[1]
    _check_tensors(hidden, h.tp, K, M, "hidden")
    _check_tensors(weight, h.tp, K, h.shard_cols, "weight")
    _check_tensors(outs, h.tp, h.V, M, "outs")
    lp = None
    if logits is not None:
        _check_tensors(logits, h.tp, h.shard_cols, M, "logits")
        lp = _ptr_array(logits)
    st = load().hg_gather_fused(h.ptr, _ptr_array(hidden), _ptr_array(weight), lp,
                                _ptr_array(outs), M, K, _stream_ptr(stream))
    _check(st, "hg_gather_fused")


def new_row_stats(M: int, device="cuda") -> torch.Tensor:
    """Device buffer for M hg_row_stats records (int32 [M, 4])."""
    return torch.zeros((M, 4), dtype=torch.int32, device=device)


def unpack_row_stats(stats: torch.Tensor) -> dict:
    """max_logit, argmax, sum_exp, logsumexp columns of an hg_row_stats buffer."""
    f = stats.view(torch.float32)
    return {"max_logit": f[:, 0], "argmax": stats[:, 1], "sum_exp": f[:, 2], "logsumexp": f[:, 3]}


def hg_gather_stats(h: Handle, shards: Sequence[torch.Tensor], outs: Sequence[torch.Tensor],
                    stats: torch.Tensor, M: int | None = None, stream=None) -> None:
    """hg_gather plus per-row sampler statistics written into `stats`
    (a buffer from new_row_stats(M))."""
    M = shards[0].shape[0] if M is None else M
    _check_tensors(shards, h.tp, h.shard_cols, M, "shards")
    _check_tensors(outs, h.tp, h.V, M, "outs")
    if not stats.is_cuda or stats.dtype != torch.int32 or tuple(stats.shape) != (M, 4) \
            or not stats.is_contiguous():
        raise ValueError("stats: need a contiguous int32 CUDA tensor [M, 4] (new_row_stats)")
    _check(load().hg_gather_stats(h.ptr, _ptr_array(shards), _ptr_array(outs), M,
                                  stats.data_ptr(), _stream_ptr(stream)), "hg_gather_stats")


def hg_sync(h: Handle, stream=None) -> None:
    _check(load().hg_sync(h.ptr, _stream_ptr(stream)), "hg_sync")


def hg_rearm(h: Handle, stream=None) -> None:
    _check(load().hg_rearm(h.ptr, _stream_ptr(stream)), "hg_rearm")


def hg_parity(h: Handle) -> int:
    return int(load().hg_parity(h.ptr))


def hg_mailbox(h: Handle, rank: int) -> tuple:
    """(device pointer, bytes) of rank's [2, cap, V] bf16 mailbox."""
    p = ctypes.c_void_p()
    n = ctypes.c_size_t()
    _check(load().hg_mailbox(h.ptr, rank, ctypes.byref(p), ctypes.byref(n)), "hg_mailbox")
    return int(p.value), int(n.value)


class _DeviceView:
    """View of library-owned device memory for torch.as_tensor (only read)."""

    def __init__(self, ptr: int, shape: tuple, typestr: str):
        self.__cuda_array_interface__ = {"shape": shape, "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


def mailbox_words(h: Handle, rank: int) -> torch.Tensor:
    """Copy of rank's mailbox as int32 words [2, cap, V / 2] (device tensor).
    Read it only while no gather of the handle is in flight."""
    ptr, nbytes = hg_mailbox(h, rank)
    shape = (2, h.cap, h.V // 2)
    assert nbytes == 4 * shape[0] * shape[1] * shape[2]
    view = torch.as_tensor(_DeviceView(ptr, shape, "<i4"), device="cuda")
    return view.clone()


def hg_launch_shape(h: Handle, M: int) -> dict:
    """Launch shape of row count M: ctas, threads, elems_per_lane, prefetch."""
    c, t, e, p = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(load().hg_launch_shape(h.ptr, M, ctypes.byref(c), ctypes.byref(t), ctypes.byref(e),
                                  ctypes.byref(p)), "hg_launch_shape")
    return {"ctas": c.value, "threads": t.value, "elems_per_lane": e.value,
            "prefetch": bool(p.value)}


TIMELINE_SLOTS = 18  # HG_TIMELINE_SLOTS: entry, after the wait, one end time per warp


def hg_timeline(h: Handle) -> tuple:
    """(records, next): a copy of the handle's timeline as an int64 device
    tensor [calls, ctas, TIMELINE_SLOTS] of %globaltimer nanoseconds (slot 0
    entry, 1 after the wait, 2 + d when warp d finished), and the index of the
    record the next call writes. Read it only while no gather is in flight."""
    p = ctypes.c_void_p()
    calls, ctas, nxt = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(load().hg_timeline(h.ptr, ctypes.byref(p), ctypes.byref(calls), ctypes.byref(ctas),
                              ctypes.byref(nxt)), "hg_timeline")
    shape = (calls.value, ctas.value, TIMELINE_SLOTS)
    view = torch.as_tensor(_DeviceView(int(p.value), shape, "<i8"), device="cuda")
    return view.clone(), nxt.value


def hg_probe_scratch_bytes(ctas: int, threads: int) -> int:
    return int(load().hg_probe_scratch_bytes(ctas, threads))


def hg_probe(kind: int, ctas: int, threads: int, scratch: torch.Tensor | None = None,
             stream=None) -> None:
    """Measurement kernels launched as the gather is (see include/hg.h):
    kind 0 empty dependent launch, 1 one-vector push/poll/copy/re-arm
    handoff, 2 arm the handoff's scratch (a device tensor of at least
    hg_probe_scratch_bytes(ctas, threads) bytes)."""
    ptr = None
    if scratch is not None:
        if not scratch.is_cuda or scratch.numel() * scratch.element_size() < \
                hg_probe_scratch_bytes(ctas, threads):
            raise ValueError("scratch: need a CUDA tensor of hg_probe_scratch_bytes bytes")
        ptr = scratch.data_ptr()
    _check(load().hg_probe(kind, ctas, threads, ptr, _stream_ptr(stream)), "hg_probe")


def hg_debug_skip_push(h: Handle, rank: int) -> None:
    _check(load().hg_debug_skip_push(h.ptr, rank), "hg_debug_skip_push")


def hg_stock_gather(shards: Sequence[torch.Tensor], outs: Sequence[torch.Tensor],
                    M: int | None = None, stream=None) -> None:
    tp = len(shards)
    M = shards[0].shape[0] if M is None else M
    W = shards[0].shape[1]
    _check_tensors(shards, tp, W, M, "shards")
    _check_tensors(outs, tp, tp * W, M, "outs")
    _check(load().hg_stock_gather(tp, W, _ptr_array(shards), _ptr_array(outs), M,
                                  _stream_ptr(stream)), "hg_stock_gather")


HG_STATIC_MAILBOX_BYTES = 24 * 1024 * 1024


def hg_gather_static(shards: Sequence[torch.Tensor], outs: Sequence[torch.Tensor],
                     M: int | None = None, status_out: torch.Tensor | None = None,
                     stream=None) -> None:
    """The gather without any allocation (libhg's hg_gather_static), for callers
    that cannot allocate device memory; its mailbox is a fixed array inside the
    library, shared by every call. shards/outs as for hg_gather; status_out, if
    given, is a one-element int32 device tensor set to 0 (ok) or 1 (a poll gave
    up) in stream order."""
    fn = load().hg_gather_static
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p),
                   ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    tp = len(shards)
    M = shards[0].shape[0] if M is None else M
    W = shards[0].shape[1]
    need = tp * M * tp * W * 2
    if need > HG_STATIC_MAILBOX_BYTES:
        raise ValueError(f"hg_gather_static: tp={tp}, M={M}, shard_cols={W} needs {need} "
                         f"bytes of mailbox, the fixed maximum is {HG_STATIC_MAILBOX_BYTES}")
    _check_tensors(shards, tp, W, M, "shards")
    _check_tensors(outs, tp, tp * W, M, "outs")
    st_ptr = None
    if status_out is not None:
        if not status_out.is_cuda or status_out.dtype != torch.int32 or status_out.numel() < 1:
            raise ValueError("status_out: need an int32 CUDA tensor with one element")
        st_ptr = status_out.data_ptr()
    _check(fn(tp, W, _ptr_array(shards), _ptr_array(outs), M, st_ptr, _stream_ptr(stream)),
           "hg_gather_static")
