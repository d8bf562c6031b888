"""Parity of the CUDA gather (through the C ABI) with the CPU oracle.

Bit-exact bar: every output word and, after every call, every mailbox word
of both parities (which must all be the sentinel again) match the oracle;
the parity sequence matches too. Inputs come from the seeded generator with
sentinel, (+0,+0) and (-0,-0) words injected, at the pages' workload shapes
(TP8, 20480-column shards = 40 KB per rank-row, V = 163840, decode row
counts) and at small shapes that span several units and a ragged tail.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from tp_vocab_logits_gb300 import hg, synth

from helpers import assert_mailboxes_armed, empty_outs, from_dev, to_dev

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_vocab_logits_gb300 import _build
    _build.build()
    oracle.build()


def run_sequence(tp, W, cap, Ms, *, rows=None, seed=7, check_mailbox_every=1, v_real=None,
                 dist="normal", scale=3.0, sent=0.02, zero=0.01, negzero=0.01, **create_kw):
    """Gather a sequence of row counts on the GPU and in the oracle; compare
    outputs word for word, mailboxes and parity after each call."""
    h = hg.hg_create(tp, W, cap, rows, **create_kw)
    og = oracle.Gather(tp, W, cap, rows)
    V = tp * W
    for i, M in enumerate(Ms):
        bits = synth.shards(seed, tp, M, W, dist=dist, scale=scale, sent_frac=sent,
                            zero_frac=zero, negzero_frac=negzero, set_index=i % 2000,
                            v_real=v_real).numpy().view(np.uint16)
        want = og.call(bits)
        shards = to_dev(bits)
        outs = empty_outs(tp, M, V)
        assert hg.hg_parity(h) == og.parity ^ 1  # oracle already flipped
        hg.hg_gather(h, shards, outs, M)
        hg.hg_sync(h)
        assert hg.hg_parity(h) == og.parity
        got = from_dev(outs)
        if not np.array_equal(got, want):
            bad = np.argwhere(got != want)
            raise AssertionError(f"call {i} (M={M}): {len(bad)} words differ, first at {bad[:5]}")
        if check_mailbox_every and (i % check_mailbox_every == 0 or i == len(Ms) - 1):
            assert_mailboxes_armed(h, hg)
    h.close()


def test_config1_tiny_golden():
    """TP=2, V=128, cap=4, M=1, three calls (parity 0, 1, 0) against the stored
    oracle values of tests/golden/config1_tiny.json."""
    with open(os.path.join(HERE, "golden", "config1_tiny.json")) as f:
        gd = json.load(f)
    tp, W, cap = gd["tp"], gd["shard_cols"], gd["cap"]
    h = hg.hg_create(tp, W, cap)
    for c in gd["calls"]:
        shards_w = np.array([[[int(x, 16) for x in row] for row in r] for r in c["shards"]],
                            dtype=np.uint32)
        want = np.array([[[int(x, 16) for x in row] for row in r] for r in c["out"]],
                        dtype=np.uint32)
        assert hg.hg_parity(h) == c["parity_before"]
        outs = empty_outs(tp, 1, tp * W)
        hg.hg_gather(h, to_dev(shards_w.view(np.uint16).reshape(tp, 1, W)), outs, 1)
        hg.hg_sync(h)
        np.testing.assert_array_equal(from_dev(outs).view(np.uint32), want)
        assert hg.hg_parity(h) == c["parity_after"]
        assert_mailboxes_armed(h, hg)
    h.close()


@pytest.mark.parametrize("tp,W,cap,Ms", [
    (2, 64, 4, [1, 1, 1]),             # config 1 shape
    (2, 8, 1, [1] * 5),                # one vector per rank-row
    (2, 4, 2, [1, 2, 2, 1]),           # V=8: word path (W % 8 != 0)
    (3, 6, 3, [3, 1, 2, 3]),           # odd TP, word path
    (4, 72, 5, [5, 4, 1, 3]),          # ragged: 9 vectors per rank-row
    (5, 1000, 3, [3, 2, 1]),           # generic-TP kernel, ragged tail of a 128-unit
    (1, 16, 2, [2, 1, 2]),             # degenerate TP=1
    (8, 1002, 4, [4, 1, 3]),           # word path, 501 words per rank-row
    (16, 4096, 4, [4, 1, 2]),          # TP16 vector path
    (8, 20480, 8, [1, 2, 3, 4, 5, 8, 8, 1]),  # decode shapes, both parities reused
])
def test_parity_vs_oracle(tp, W, cap, Ms):
    run_sequence(tp, W, cap, Ms)


@pytest.mark.parametrize("vpt,ctas,pref,coop", [
    (1, 1, 0, False), (1, 3, 1, False), (2, 7, 1, False), (4, 2, 2, False), (2, 0, 1, False),
    (4, 0, 0, False), (1, 1, 1, False), (3, 0, 0, False), (3, 5, 1, False), (5, 4, 1, False),
    (6, 0, 0, False), (6, 2, 1, False), (1, 0, 0, True), (4, 5, 1, True), (3, 0, 0, True),
    (0, 0, 0, True)])
def test_launch_shapes_vs_oracle(vpt, ctas, pref, coop):
    """Forced launch shapes: small grids make every CTA loop over many units (a
    single CTA consumes its own pushes one iteration later); with and without
    the shard prefetch; cooperative and programmatic-dependent launches."""
    run_sequence(4, 2048, 6, [6, 1, 5, 6], elems_per_lane=vpt, ctas=ctas, prefetch=pref,
                 cooperative=coop)
    h = hg.hg_create(4, 2048, 6, elems_per_lane=vpt, ctas=ctas, prefetch=pref)
    assert hg.hg_launch_shape(h, 6)["prefetch"] == (pref == 1)
    h.close()


@pytest.mark.parametrize("vpt,ctas,pref", [(3, 0, 0), (5, 0, 0), (6, 2, 1), (5, 3, 1), (1, 0, 0)])
def test_word_path_shapes_vs_oracle(vpt, ctas, pref):
    """4-byte word path (W % 8 != 0: 499 words per rank-row, ragged for every
    unit size) with forced elements per lane, grids and prefetch."""
    run_sequence(3, 998, 4, [4, 1, 3, 2], elems_per_lane=vpt, ctas=ctas, prefetch=pref)


def test_multi_wave_decode_width_vs_oracle():
    """TP8, V=163840, M=64: more units than co-resident CTAs, so every CTA loops
    over units; three calls (both parities) against the oracle word for word."""
    tp, W, M = 8, 20480, 64
    h = hg.hg_create(tp, W, M)
    shape = hg.hg_launch_shape(h, M)
    units = M * tp * -(-(W // 8) // (32 * shape["elems_per_lane"]))
    assert shape["ctas"] < units
    h.close()
    run_sequence(tp, W, M, [M, M, M])


def _back_to_back(h, og, tp, W, Ms, seed):
    """Issue every call of Ms on one stream with no synchronisation between
    them (each into its own outputs), then compare all of them with the
    oracle run through the same sequence."""
    wants, outs_all = [], []
    for i, M in enumerate(Ms):
        bits = synth.shards(seed, tp, M, W, scale=3.0, sent_frac=0.01, set_index=i) \
            .numpy().view(np.uint16)
        wants.append(og.call(bits))
        outs = empty_outs(tp, M, tp * W)
        hg.hg_gather(h, to_dev(bits), outs, M)
        outs_all.append(outs)
    hg.hg_sync(h)
    assert hg.hg_parity(h) == og.parity
    for i, (want, outs) in enumerate(zip(wants, outs_all)):
        got = from_dev(outs)
        if not np.array_equal(got, want):
            raise AssertionError(f"call {i} (M={Ms[i]}): {int((got != want).sum())} words differ")
    assert_mailboxes_armed(h, hg)


def test_varying_rows_back_to_back():
    """TP8, V=163840: row counts 1, 1, 1, 2, 8, 3, 5, 4, 1, 8, 2 issued back to
    back on one handle (each call's launch overlapping the previous one's
    tail), synchronised only at the end; single-wave and looping grids
    alternate from call to call."""
    tp, W, cap = 8, 20480, 8
    h = hg.hg_create(tp, W, cap)
    og = oracle.Gather(tp, W, cap)
    _back_to_back(h, og, tp, W, [1, 1, 1, 2, 8, 3, 5, 4, 1, 8, 2], seed=11)
    h.close()


def test_autotuned_shapes_vs_oracle():
    """hg_options.autotune at the decode width (TP8, V=163840, the speculative
    row counts): the tuned shapes are valid launch shapes, the parity starts at
    0, and a seeded sequence of calls issued back to back matches the oracle;
    the same with the parity on the device."""
    tp, W, cap = 8, 20480, 8
    rows = [1, 2, 3, 4, 5, 8]
    for dp in (False, True):
        h = hg.hg_create(tp, W, cap, rows, autotune=True, device_parity=dp)
        assert hg.hg_parity(h) == 0
        for M in rows:
            s = hg.hg_launch_shape(h, M)
            assert 1 <= s["elems_per_lane"] <= 6 and s["ctas"] >= 1
            assert s["threads"] == 32 * tp
        og = oracle.Gather(tp, W, cap, rows)
        _back_to_back(h, og, tp, W, synth.row_sequence(5, 14, rows), seed=12 + dp)
        h.close()


def test_autotune_honours_forced_fields():
    """Autotuning with elements per lane, CTAs and prefetch forced keeps them."""
    h = hg.hg_create(4, 2048, 6, autotune=True, elems_per_lane=2, ctas=3, prefetch=1)
    for M in range(1, 7):
        s = hg.hg_launch_shape(h, M)
        assert s["elems_per_lane"] == 2 and s["ctas"] == 3 and s["prefetch"]
    h.close()
    run_sequence(4, 2048, 6, [6, 1, 5], autotune=True)


@pytest.mark.parametrize("tp", [24, 32])
def test_wide_tp_vs_oracle(tp):
    """TP above 16 runs 1024-thread CTAs (one warp per rank)."""
    run_sequence(tp, 256, 3, [3, 1, 2])


def test_config2_decode_m1():
    """TP8, V=163840, cap=8, M=1: 1000 calls back to back on one stream with
    0.1 % sentinel words (and, beyond the workload's recipe, 0.1 % of the
    generator's other classes next to the sentinel), rotating three input
    sets; every call's outputs against the oracle word for word (each call
    gathers into its own slot of a ring of outputs, checked once the ring is
    full), mailboxes at the end."""
    tp, W, cap, calls, ring = 8, 20480, 8, 1000, 50
    h = hg.hg_create(tp, W, cap)
    og = oracle.Gather(tp, W, cap)
    sets = [synth.shards(1, tp, 1, W, scale=3.0, sent_frac=0.001, extra_frac=0.001, set_index=i)
            .numpy().view(np.uint16) for i in range(3)]
    dev = [to_dev(s) for s in sets]
    outs = [empty_outs(tp, 1, tp * W) for _ in range(ring)]
    wants = []
    for i in range(calls):
        wants.append(og.call(sets[i % 3]))
        hg.hg_gather(h, dev[i % 3], outs[i % ring], 1)
        if i % ring == ring - 1 or i == calls - 1:
            hg.hg_sync(h)
            for k, want in enumerate(wants):
                got = from_dev(outs[(i - len(wants) + 1 + k) % ring])
                if not np.array_equal(got, want):
                    raise AssertionError(f"call {i - len(wants) + 1 + k}: outputs differ")
            wants = []
    assert hg.hg_parity(h) == og.parity
    assert_mailboxes_armed(h, hg)
    h.close()


def test_config3_speculative_padded_vocab():
    """TP8, real vocab 163837 padded to 163840 (pads = bf16 -inf), 1000 calls
    whose row counts follow a seeded sequence over {1,2,3,4,5,8}, cap 8; every
    call against the oracle word for word, pads checked, the padded-vocab
    slice checked on a rank per call; mailboxes checked every 100 calls."""
    tp, W, cap, v_real = 8, 20480, 8, 163837
    rows = [1, 2, 3, 4, 5, 8]
    Ms = synth.row_sequence(2, 1000, rows)
    h = hg.hg_create(tp, W, cap, rows)
    og = oracle.Gather(tp, W, cap, rows)
    for i, M in enumerate(Ms):
        bits = synth.shards(2, tp, M, W, scale=3.0, set_index=i, v_real=v_real) \
            .numpy().view(np.uint16)
        want = og.call(bits)
        outs = empty_outs(tp, M, tp * W)
        hg.hg_gather(h, to_dev(bits), outs, M)
        hg.hg_sync(h)
        got = from_dev(outs)
        if not np.array_equal(got, want):
            raise AssertionError(f"call {i} (M={M}): outputs differ")
        assert (got[:, :, v_real:] == 0xFF80).all()
        d = i % tp
        sliced = outs[d][:, :v_real]
        np.testing.assert_array_equal(sliced.cpu().numpy().view(np.uint16),
                                      oracle.slice_vocab(want[d], v_real))
        if i % 100 == 99:
            assert_mailboxes_armed(h, hg)
    assert_mailboxes_armed(h, hg)
    h.close()


@pytest.mark.parametrize("tp,W,M", [(2, 4096, 64), (4, 8192, 32), (8, 20480, 8),
                                    (2, 65536, 8)])
def test_config4_small_points_vs_oracle(tp, W, M):
    """Bandwidth-sweep points the oracle finishes quickly, cap = M, U(-20, 20)."""
    run_sequence(tp, W, M, [M, M, M], dist="uniform", scale=20.0, sent=0.0, zero=0.0,
                 negzero=0.0, seed=3)


def _host_bytes_available() -> int:
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    return 0


@pytest.mark.parametrize("tp,W,M", [(8, 20480, 64), (8, 20480, 256), (16, 65536, 64),
                                    (16, 4096, 256), (4, 65536, 128)])
def test_config4_large_points_vs_oracle(tp, W, M):
    """Full-size sweep points (cap = M, U(-20, 20), with 0.1 % sentinel words
    and 0.1 % of the other classes next to it): every output word of every
    rank against the oracle run through the same three calls (both parities),
    and every mailbox re-armed, as the oracle's are. The oracle holds every
    rank's two-parity mailbox in host memory (up to 4.3 GB, at TP16 with
    65536-column shards and M=64); a point whose oracle state would not fit in
    the host's available memory is skipped, and says so."""
    V = tp * W
    need = tp * 2 * M * V * 2 + 2 * tp * M * V * 2 + tp * M * W * 2
    avail = _host_bytes_available()
    if 1.5 * need > avail:
        pytest.skip(f"the oracle needs {need / 2**30:.1f} GiB of host memory, "
                    f"{avail / 2**30:.1f} GiB available")
    h = hg.hg_create(tp, W, M)
    og = oracle.Gather(tp, W, M)
    outs = empty_outs(tp, M, V)
    for i in range(3):
        bits = synth.shards(3, tp, M, W, dist="uniform", scale=20.0, sent_frac=0.001,
                            extra_frac=0.001, set_index=i, device="cuda")
        want = og.call(bits.cpu().numpy().view(np.uint16))
        hg.hg_gather(h, [bits[r] for r in range(tp)], outs, M)
        hg.hg_sync(h)
        assert hg.hg_parity(h) == og.parity
        for d in range(tp):
            got = outs[d].cpu().numpy().view(np.uint16)
            if not np.array_equal(got, want[d]):
                raise AssertionError(f"call {i} rank {d}: "
                                     f"{int((got != want[d]).sum())} bf16 columns differ")
        del want
    assert_mailboxes_armed(h, hg)
    h.close()


@pytest.mark.parametrize("shards_on_host", [True, False])
def test_host_buffers_vs_oracle(shards_on_host):
    """hg_gather_host at the decode width (TP8, V=163840): outputs in
    page-locked host memory written by the kernel itself, shards in host or
    device memory; every call against the oracle, both parities, rows 1..3."""
    tp, W, cap = 8, 20480, 4
    h = hg.hg_create(tp, W, cap)
    og = oracle.Gather(tp, W, cap)
    for i, M in enumerate([1, 3, 2, 1]):
        bits = synth.shards(21, tp, M, W, scale=3.0, sent_frac=0.01, set_index=i) \
            .numpy().view(np.uint16)
        want = og.call(bits)
        host_sh = [torch.from_numpy(bits[r].view(np.int16).copy()).pin_memory()
                   for r in range(tp)]
        shards = host_sh if shards_on_host else [t.cuda() for t in host_sh]
        outs = [torch.full((M, tp * W), 7, dtype=torch.int16).pin_memory() for _ in range(tp)]
        hg.hg_gather_host(h, shards, outs, M)
        hg.hg_sync(h)
        got = np.stack([o.numpy().view(np.uint16) for o in outs])
        np.testing.assert_array_equal(got, want)
        assert hg.hg_parity(h) == og.parity
    assert_mailboxes_armed(h, hg)
    h.close()


def test_host_buffers_rejects_pageable_memory():
    """Pageable host memory (not page-locked) is refused before any device
    work, with no parity flip; the binding refuses it before the call."""
    import ctypes
    tp, W = 2, 64
    h = hg.hg_create(tp, W, 2)
    lib = hg.load()
    pageable = [np.zeros((1, W), np.int16) for _ in range(tp)]
    outs_p = [np.zeros((1, tp * W), np.int16) for _ in range(tp)]
    sp = (ctypes.c_void_p * tp)(*[a.ctypes.data for a in pageable])
    op = (ctypes.c_void_p * tp)(*[a.ctypes.data for a in outs_p])
    assert lib.hg_gather_host(h.ptr, sp, op, 1, None) == hg.HG_ERR_ARG
    assert hg.hg_parity(h) == 0
    with pytest.raises(ValueError):
        hg.hg_gather_host(h, [torch.zeros(1, W, dtype=torch.int16) for _ in range(tp)],
                          [torch.zeros(1, tp * W, dtype=torch.int16).pin_memory()
                           for _ in range(tp)], 1)
    hg.hg_sync(h)
    h.close()


def test_stock_baseline_matches_concat():
    """The cudaMemcpy2D baseline is the plain concat; without sentinel words it
    equals the gather bit for bit."""
    tp, W, M = 8, 20480, 4
    bits = synth.shards(5, tp, M, W, scale=3.0).numpy().view(np.uint16)
    shards = to_dev(bits)
    a = empty_outs(tp, M, tp * W)
    b = empty_outs(tp, M, tp * W)
    hg.hg_stock_gather(shards, a, M)
    h = hg.hg_create(tp, W, 8)
    hg.hg_gather(h, shards, b, M)
    hg.hg_sync(h)
    cat = np.concatenate([bits[r] for r in range(tp)], axis=1)
    for d in range(tp):
        np.testing.assert_array_equal(a[d].cpu().numpy().view(np.uint16), cat)
        assert torch.equal(a[d], b[d])
    h.close()


def test_rejected_calls_change_nothing():
    """Unserved row counts (M = 0, M > cap, M not in rows), misaligned or
    missing pointers and graph capture are refused before any device work:
    parity, mailboxes and outputs stay as they were."""
    tp, W, cap = 4, 64, 4
    h = hg.hg_create(tp, W, cap, rows=[1, 3])
    bits = synth.shards(9, tp, 3, W, scale=3.0).numpy().view(np.uint16)
    shards = to_dev(bits)
    outs = empty_outs(tp, 3, tp * W)
    lib = hg.load()
    sp = hg._ptr_array(shards)
    op = hg._ptr_array(outs)
    stream = torch.cuda.current_stream().cuda_stream
    for M in (0, 2, 4, 5, -1):
        assert lib.hg_gather(h.ptr, sp, op, M, stream) == hg.HG_ERR_ROWS
    # misaligned output pointer (2 bytes off) and a NULL shard pointer
    import ctypes
    bad = (ctypes.c_void_p * tp)(*[o.data_ptr() + 2 for o in outs])
    assert lib.hg_gather(h.ptr, sp, bad, 3, stream) == hg.HG_ERR_ARG
    nul = (ctypes.c_void_p * tp)(*([None] + [s.data_ptr() for s in shards[1:]]))
    assert lib.hg_gather(h.ptr, nul, op, 3, stream) == hg.HG_ERR_ARG
    assert lib.hg_gather(None, sp, op, 3, stream) == hg.HG_ERR_ARG
    # graph capture: refused, nothing captured
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.capture_begin()
        st = lib.hg_gather(h.ptr, sp, op, 3, s.cuda_stream)
        g.capture_end()
    assert st == hg.HG_ERR_CAPTURE
    torch.cuda.synchronize()
    assert hg.hg_parity(h) == 0
    assert (from_dev(outs) == 0x5A5A).all()
    assert_mailboxes_armed(h, hg)
    # a served call still works and is the first use of parity 0
    og = oracle.Gather(tp, W, cap, [1, 3])
    hg.hg_gather(h, shards, outs, 3)
    hg.hg_sync(h)
    np.testing.assert_array_equal(from_dev(outs), og.call(bits))
    h.close()


def test_create_rejects_bad_sizes():
    for args in [(0, 64, 4), (hg.HG_MAX_TP + 1, 64, 4), (2, 7, 4), (2, 0, 4),
                 (2, 64, 0)]:
        with pytest.raises(hg.HGError) as e:
            hg.hg_create(*args)
        assert e.value.status == hg.HG_ERR_ARG
    with pytest.raises(hg.HGError):
        hg.hg_create(2, 64, 4, rows=[5])
    for kw in ({"elems_per_lane": 7}, {"elems_per_lane": -1}, {"prefetch": 3}, {"ctas": -2}):
        with pytest.raises(hg.HGError) as e:
            hg.hg_create(2, 64, 4, **kw)
        assert e.value.status == hg.HG_ERR_ARG
    with pytest.raises(hg.HGError):
        hg.hg_create(24, 64, 4, elems_per_lane=3)  # 1024-thread CTAs: 1 or 2 per lane
    h = hg.hg_create(8, 20480, 8)
    # from four rows on, the width whose busiest SM moves the fewest vectors:
    # M=4 6 per lane (576 against 640), M=5 and M=6 4, M=7 and M=8 5
    Ms = (1, 2, 3, 4, 5, 6, 7, 8)
    shapes = [hg.hg_launch_shape(h, M) for M in Ms]
    assert [s["elems_per_lane"] for s in shapes] == [3, 3, 3, 6, 4, 4, 5, 5]
    assert [s["ctas"] for s in shapes] == [216, 432, 608, 448, 608, 608, 608, 608]
    h.close()
    # the same count on other shapes of the bandwidth sweep (each measured faster):
    # TP4 W=20480 M=8 6 per lane on 448 CTAs, TP2 W=20480 M=32 5 per lane
    for tp, W, M, want in [(4, 20480, 8, (448, 6)), (2, 20480, 32, (1024, 5))]:
        h = hg.hg_create(tp, W, M, rows=[M])
        s = hg.hg_launch_shape(h, M)
        assert (s["ctas"], s["elems_per_lane"]) == want, (tp, W, M, s)
        h.close()
    h = hg.hg_create(16, 4096, 2)
    assert hg.hg_launch_shape(h, 1)["elems_per_lane"] == 4
    h.close()


def test_timeout_recovery():
    """Failure detection without a GPU fault: rank 3's push is skipped (host
    test hook), the other ranks' polls give up after 20 ms, hg_sync reports
    the timeout, later calls are refused until hg_rearm, and after re-arming
    the gather is exact again."""
    tp, W, cap = 8, 4096, 2
    h = hg.hg_create(tp, W, cap, poll_timeout_ns=20_000_000)
    bits = synth.shards(6, tp, 2, W, scale=3.0, sent_frac=0.01).numpy().view(np.uint16)
    shards = to_dev(bits)
    outs = empty_outs(tp, 2, tp * W)
    hg.hg_debug_skip_push(h, 3)
    hg.hg_gather(h, shards, outs, 2)
    with pytest.raises(hg.HGError) as e:
        hg.hg_sync(h)
    assert e.value.status == hg.HG_ERR_TIMEOUT
    with pytest.raises(hg.HGError) as e:
        hg.hg_gather(h, shards, outs, 2)
    assert e.value.status == hg.HG_ERR_STATE
    hg.hg_debug_skip_push(h, -1)
    hg.hg_rearm(h)
    assert hg.hg_parity(h) == 0
    assert_mailboxes_armed(h, hg)
    og = oracle.Gather(tp, W, cap)
    for _ in range(3):
        want = og.call(bits)
        hg.hg_gather(h, shards, outs, 2)
        hg.hg_sync(h)
        np.testing.assert_array_equal(from_dev(outs), want)
    assert_mailboxes_armed(h, hg)
    h.close()


@pytest.mark.parametrize("tp,W,n_calls,kw", [
    (8, 20480, 301, {}),
    (8, 20480, 101, {"device_parity": True}),
    (4, 4096, 201, {}),
])
def test_chain_reads_the_previous_kernels_output(tp, W, n_calls, kw):
    """Each call's shards are slices of the previous call's outputs, so the
    previous gather kernel is still writing them when the next call's launch
    begins (programmatic dependent launch) and prefetches them into L2. Every
    value read must still be the previous call's result. Two output sets
    alternate; call i reads set (i - 1) % 2 and writes set i % 2, and rank r's
    shard is segment (r + shift) % tp of rank r's row, with shift 1 when
    reading set 0 and 2 when reading set 1: a read of the set's older contents
    (two calls back) would show a rotation of 3 segments. The final outputs
    are compared with the oracle run through the same chain."""
    h = hg.hg_create(tp, W, 1, **kw)
    og = oracle.Gather(tp, W, 1)
    bits = synth.shards(41, tp, 1, W, scale=3.0, sent_frac=0.01).numpy().view(np.uint16)
    bufs = [empty_outs(tp, 1, tp * W), empty_outs(tp, 1, tp * W)]
    shifts = (1, 2)

    def seg(row, r, src):
        k = (r + shifts[src]) % tp
        return row[:, k * W:(k + 1) * W]

    calls = [hg.GatherCall(h, [seg(bufs[src][r], r, src) for r in range(tp)], bufs[1 - src], 1)
             for src in (0, 1)]
    hg.GatherCall(h, to_dev(bits), bufs[0], 1)()
    for i in range(1, n_calls):
        calls[(i - 1) % 2]()
    hg.hg_sync(h)

    want = og.call(bits)
    for i in range(1, n_calls):
        src = (i - 1) % 2
        want = og.call(np.ascontiguousarray(np.stack([seg(want[r], r, src) for r in range(tp)])))
    np.testing.assert_array_equal(from_dev(bufs[(n_calls - 1) % 2]), want)
    assert_mailboxes_armed(h, hg)
    h.close()
