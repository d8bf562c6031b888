"""hg_gather_static: the gather for callers that cannot allocate device memory
(a serving engine whose allocator already holds the GPU's free memory, a
plug-in that must not allocate outside its host's allocator, a loop that cannot
pay for cudaMalloc's implicit synchronisation). Its mailbox is a fixed array
inside the library, shared by every call.

Called through the C ABI, two calls in a row, its outputs must equal hg_gather's
on the same shards bit for bit (the gather is exact). This file is collected
last so that a run that stops at the first failure has run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from tp_vocab_logits_gb300 import _build, hg, synth

pytestmark = pytest.mark.gpu


def _c_gather_static(lib, tp, W, shards, outs, M, status, stream):
    fn = lib.hg_gather_static
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p),
                   ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    sp = (ctypes.c_void_p * tp)(*[s.data_ptr() for s in shards])
    op = (ctypes.c_void_p * tp)(*[o.data_ptr() for o in outs])
    return fn(tp, W, sp, op, M, status.data_ptr() if status is not None else None, stream)


def test_static_gather_matches_handle_gather():
    _build.build()
    lib = hg.load()
    tp, W = 8, 20480
    stream = torch.cuda.current_stream().cuda_stream
    h = hg.hg_create(tp, W, 8)
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    for call, M in enumerate([2, 3]):
        bits = synth.shards(11, tp, M, W, scale=3.0, sent_frac=0.01, zero_frac=0.01,
                            negzero_frac=0.01, set_index=call, device="cuda")
        shards = [bits[r] for r in range(tp)]
        ref = [torch.empty((M, tp * W), dtype=torch.int16, device="cuda") for _ in range(tp)]
        got = [torch.full((M, tp * W), 0x1234, dtype=torch.int16, device="cuda")
               for _ in range(tp)]
        hg.hg_gather(h, shards, ref, M)
        assert _c_gather_static(lib, tp, W, shards, got, M, status, stream) == hg.HG_OK
        torch.cuda.synchronize()
        hg.hg_sync(h)
        assert status.item() == 0
        for d in range(tp):
            assert torch.equal(got[d], ref[d]), f"call {call}, rank {d}"
    h.close()


def test_static_gather_shapes_in_sequence():
    """The shared array across calls of different shapes, back to back: the
    16-byte vector path (TP8, V=163840, up to the largest M that fits, 9), the
    4-byte word path (TP=2, shard width 6; TP=4, width 1000), and 1024-thread
    CTAs (TP=32). Each call re-arms only the region it uses, so a smaller call
    right after a larger one must not see the larger call's leftovers; every
    call's outputs equal hg_gather's on the same shards."""
    _build.build()
    lib = hg.load()
    stream = torch.cuda.current_stream().cuda_stream
    seq = [(8, 20480, 9), (2, 6, 1), (32, 256, 3), (8, 20480, 1), (2, 6, 5), (4, 1000, 7),
           (32, 256, 1), (8, 20480, 4)]
    handles = {}
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    for call, (tp, W, M) in enumerate(seq):
        assert tp * M * tp * W * 2 <= hg.HG_STATIC_MAILBOX_BYTES
        if (tp, W) not in handles:
            handles[(tp, W)] = hg.hg_create(tp, W, 9)
        h = handles[(tp, W)]
        bits = synth.shards(12, tp, M, W, scale=3.0, sent_frac=0.02, zero_frac=0.01,
                            negzero_frac=0.01, set_index=call, device="cuda")
        shards = [bits[r] for r in range(tp)]
        ref = [torch.empty((M, tp * W), dtype=torch.int16, device="cuda") for _ in range(tp)]
        got = [torch.full((M, tp * W), 0x1234, dtype=torch.int16, device="cuda")
               for _ in range(tp)]
        hg.hg_gather(h, shards, ref, M)
        assert _c_gather_static(lib, tp, W, shards, got, M, status, stream) == hg.HG_OK
        torch.cuda.synchronize()
        hg.hg_sync(h)
        assert status.item() == 0, f"call {call}"
        for d in range(tp):
            assert torch.equal(got[d], ref[d]), f"call {call} (tp={tp}, W={W}, M={M}), rank {d}"
    for h in handles.values():
        h.close()


def test_static_gather_rejects_oversize_without_device_work():
    _build.build()
    lib = hg.load()
    tp, W = 8, 20480
    M = hg.HG_STATIC_MAILBOX_BYTES // (tp * tp * W * 2) + 1  # one row too many
    shards = [torch.zeros((1, W), dtype=torch.int16, device="cuda") for _ in range(tp)]
    outs = [torch.full((1, tp * W), 5, dtype=torch.int16, device="cuda") for _ in range(tp)]
    stream = torch.cuda.current_stream().cuda_stream
    assert _c_gather_static(lib, tp, W, shards, outs, M, None, stream) == hg.HG_ERR_ARG
    torch.cuda.synchronize()
    assert all(bool((o == 5).all()) for o in outs)
    with pytest.raises(ValueError):
        hg.hg_gather_static(shards, outs, M)
