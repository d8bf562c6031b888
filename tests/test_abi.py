"""The C ABI library loads without a GPU, exports every entry point that
include/hg.h declares, and its host-side argument checks answer without
touching the device."""

import ctypes
import os
import re

import pytest
import torch

from tp_vocab_logits_gb300 import _build, hg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return hg.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                src = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(hg_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ["hg_create", "hg_gather", "hg_destroy", "hg_sync", "hg_rearm", "hg_parity",
              "hg_mailbox", "hg_stock_gather", "hg_strerror"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"libhg.so does not export {name}"


def test_host_checks_without_device(lib):
    out = ctypes.c_void_p()
    for tp, W, cap in [(0, 64, 4), (hg.HG_MAX_TP + 1, 64, 4), (2, 7, 4), (2, 0, 4), (2, 64, 0)]:
        assert lib.hg_create(tp, W, cap, None, 0, ctypes.byref(out)) == hg.HG_ERR_ARG
        assert out.value is None
    rows = (ctypes.c_int * 2)(1, 9)
    assert lib.hg_create(2, 64, 4, rows, 2, ctypes.byref(out)) == hg.HG_ERR_ARG
    assert lib.hg_create(2, 64, 4, None, 0, None) == hg.HG_ERR_ARG
    assert lib.hg_gather(None, None, None, 1, None) == hg.HG_ERR_ARG
    assert lib.hg_gather_host(None, None, None, 1, None) == hg.HG_ERR_ARG
    assert lib.hg_sync(None, None) == hg.HG_ERR_ARG
    assert lib.hg_rearm(None, None) == hg.HG_ERR_ARG
    assert lib.hg_parity(None) == -1
    assert lib.hg_destroy(None) == hg.HG_OK
    assert lib.hg_debug_skip_push(None, 0) == hg.HG_ERR_ARG
    c = ctypes.c_int()
    assert lib.hg_launch_shape(None, 1, ctypes.byref(c), None, None, None) == hg.HG_ERR_ARG
    assert lib.hg_stock_gather(0, 8, None, None, 1, None) == hg.HG_ERR_ARG
    p = ctypes.c_void_p()
    assert lib.hg_timeline(None, ctypes.byref(p), None, None, None) == hg.HG_ERR_ARG
    for kind, ctas, threads in [(3, 1, 32), (-1, 1, 32), (0, 0, 32), (0, 1, 33), (0, 1, 1024)]:
        assert lib.hg_probe(kind, ctas, threads, None, None) == hg.HG_ERR_ARG
    assert lib.hg_probe(1, 4, 64, None, None) == hg.HG_ERR_ARG   # scratch needed
    assert lib.hg_probe_scratch_bytes(4, 64) == 2 * 4 * 64 * 16 + 16
    assert lib.hg_probe_scratch_bytes(0, 64) == 0
    for code in range(7):
        assert lib.hg_strerror(code)
    assert lib.hg_strerror(99) == b"unknown status"


def test_direct_call_object_marshals_and_raises(lib):
    """The _hgcall extension builds and loads, holds the pointer lists, calls
    the C entry point and turns a failed status into HGError: here a closed
    handle (NULL), which hg_gather rejects before any CUDA call."""
    mod = hg._pycall()

    class Closed:
        ptr = None

    fn = ctypes.cast(lib.hg_gather, ctypes.c_void_p).value
    raised = []

    def on_error(status):
        raised.append(status)
        raise hg.HGError(status, "hg_gather")

    call = mod.Call(fn, Closed(), [16, 32], [48, 64], 1, 0, None, on_error)
    with pytest.raises(hg.HGError):
        call()
    assert raised == [hg.HG_ERR_ARG]
    with pytest.raises(TypeError):
        call(1)
    with pytest.raises(ValueError):
        mod.Call(fn, Closed(), [16, 32], [48], 1, 0, None, on_error)


def test_binding_rejects_bad_tensor_lists_before_the_library():
    """GatherCall checks the tensor lists before anything reaches libhg: a
    list of the wrong length, and host tensors that are not page-locked (the
    kernel can only read and write host memory that is). The dtype and shape
    checks after these need page-locked or device tensors; the GPU tests
    cover them (test_rejected_calls_change_nothing)."""
    h = hg.Handle(0, 2, 8, 1, None)  # never handed to the library here
    shards = [torch.zeros(1, 8, dtype=torch.int16) for _ in range(2)]
    outs = [torch.zeros(1, 16, dtype=torch.int16) for _ in range(2)]
    with pytest.raises(ValueError, match="expected 2 tensors"):
        hg.GatherCall(h, shards[:1], outs, 1)
    with pytest.raises(ValueError, match="page-locked"):
        hg.GatherCall(h, shards, outs, 1)
