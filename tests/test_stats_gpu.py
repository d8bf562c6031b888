"""Sampler statistics of the gathered rows (hg_gather_stats): each unit folded
where it is pushed, the cells reduced per row in the same kernel.

Per gathered row: max_logit and argmax must equal the oracle exactly (the max
of bf16 values is exact in fp32, and both sides resolve ties to the smallest
column); sum_exp, accumulated in fp32 with the fast exponential, within a
relative 1e-4 of the oracle's float64 sum (a few ulp per term over per-lane
runs of at most 48 terms, then runs of at most 8 cells and pairwise
folding); logsumexp within 1e-4 absolute. The gathered outputs themselves stay
bit-exact."""

import numpy as np
import pytest
import torch

import oracle
from tp_vocab_logits_gb300 import hg, synth

from helpers import assert_mailboxes_armed, empty_outs, from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_vocab_logits_gb300 import _build
    _build.build()
    oracle.build()


def check(h, og, bits, M):
    tp, V = h.tp, h.V
    want = og.call(bits)
    outs = empty_outs(tp, M, V)
    st = hg.new_row_stats(M)
    hg.hg_gather_stats(h, to_dev(bits), outs, st, M)
    hg.hg_sync(h)
    np.testing.assert_array_equal(from_dev(outs), want)
    got = {k: v.cpu().numpy() for k, v in hg.unpack_row_stats(st).items()}
    for m in range(M):
        mx, arg, se = oracle.row_stats(want[0][m])
        assert got["max_logit"][m] == mx, (m, got["max_logit"][m], mx)
        assert got["argmax"][m] == arg, (m, got["argmax"][m], arg)
        if se == 0.0:
            assert got["sum_exp"][m] == 0.0 and got["logsumexp"][m] == -np.inf
        else:
            assert abs(got["sum_exp"][m] - se) <= 1e-4 * se, (m, got["sum_exp"][m], se)
            assert abs(got["logsumexp"][m] - (mx + np.log(se))) <= 1e-4
    assert_mailboxes_armed(h, hg)


@pytest.mark.parametrize("M", [1, 3, 8])
def test_stats_decode_shapes(M):
    """TP8, V=163840 padded from 163837 (pads -inf), sentinel words injected,
    two calls (both parities, statistics cells reused)."""
    tp, W = 8, 20480
    h = hg.hg_create(tp, W, 8)
    og = oracle.Gather(tp, W, 8)
    for i in range(2):
        bits = synth.shards(31, tp, M, W, scale=3.0, sent_frac=0.01, negzero_frac=0.01,
                            set_index=i, v_real=163837).numpy().view(np.uint16)
        check(h, og, bits, M)
    h.close()


def test_stats_ties_and_special_rows():
    """Row 0: the max appears in three ranks' shards (smallest column wins);
    row 1: every value -inf; row 2: all values equal (sum = V)."""
    tp, W, M = 4, 64, 3
    h = hg.hg_create(tp, W, 4)
    og = oracle.Gather(tp, W, 4)
    bits = synth.shards(32, tp, M, W, scale=1.0).numpy().view(np.uint16).copy()
    tb = torch.tensor([30.0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]
    bits[3, 0, 5] = tb
    bits[1, 0, 60] = tb
    bits[2, 0, 7] = tb
    bits[:, 1, :] = 0xFF80
    bits[:, 2, :] = 0x3F80  # 1.0
    check(h, og, bits, M)
    h.close()


@pytest.mark.parametrize("tp,W,cap,Ms,kw", [
    (3, 6, 3, [3, 1], {}),                                 # word path (W % 8 != 0)
    (4, 2048, 6, [6, 2], {"ctas": 3, "prefetch": 1}),      # many units per CTA
    (16, 4096, 2, [2], {}),
    (8, 20480, 8, [8, 1], {"device_parity": True}),
    (1, 64, 2, [2, 1], {}),                                # degenerate TP=1
    (8, 20480, 2, [2, 1], {"elems_per_lane": 1}),          # 640 cells a row: 3 reducer batches
    (8, 20480, 2, [1, 2], {"elems_per_lane": 4}),          # the VPT 4 kernel at decode sizes
    (16, 65536, 1, [1], {"elems_per_lane": 5}),            # 6-cell batches, 832 cells: 5 batches
    (4, 6144, 3, [3], {"elems_per_lane": 6}),
])
def test_stats_shapes(tp, W, cap, Ms, kw):
    h = hg.hg_create(tp, W, cap, **kw)
    og = oracle.Gather(tp, W, cap)
    for i, M in enumerate(Ms):
        bits = synth.shards(33, tp, M, W, scale=4.0, sent_frac=0.02, set_index=i) \
            .numpy().view(np.uint16)
        check(h, og, bits, M)
    h.close()


def test_stats_interleaved_with_plain_gathers():
    """Plain and statistics calls on one handle share the parity sequence."""
    tp, W = 8, 4096
    h = hg.hg_create(tp, W, 4)
    og = oracle.Gather(tp, W, 4)
    for i, M in enumerate([2, 1, 4, 3]):
        bits = synth.shards(34, tp, M, W, scale=3.0, set_index=i).numpy().view(np.uint16)
        if i % 2:
            check(h, og, bits, M)
        else:
            want = og.call(bits)
            outs = empty_outs(tp, M, tp * W)
            hg.hg_gather(h, to_dev(bits), outs, M)
            hg.hg_sync(h)
            np.testing.assert_array_equal(from_dev(outs), want)
    h.close()


@pytest.mark.parametrize("device_parity", [False, True])
def test_stats_back_to_back_random_rows(device_parity):
    """A stream of 1,500 calls with a seeded sequence of row counts, two in
    three with statistics and one in three plain, on one handle, synchronised
    every 64 calls: every output row and every statistics row against the
    oracle. Consecutive calls reuse each cell and mailbox row across parities
    and shapes, which is where a missing re-arm or a cell read too early would
    show."""
    tp, W, cap, n_calls, ring = 8, 20480, 8, 1500, 64
    h = hg.hg_create(tp, W, cap, device_parity=device_parity)
    sets, want_dev, want_stats = [], [], []
    for i in range(8):
        bits = synth.shards(92, tp, cap, W, scale=3.0, sent_frac=0.01, set_index=i) \
            .numpy().view(np.uint16)
        want = oracle.Gather(tp, W, cap).call(bits)
        sets.append(to_dev(bits))
        want_dev.append(torch.from_numpy(want[0].view(np.int16).copy()).cuda())
        want_stats.append([oracle.row_stats(want[0][m]) for m in range(cap)])
    outs = [empty_outs(tp, cap, tp * W) for _ in range(ring)]
    stats = [hg.new_row_stats(cap) for _ in range(ring)]
    Ms = synth.row_sequence(11 + device_parity, n_calls, list(range(1, cap + 1)))
    pend = []
    for i, M in enumerate(Ms):
        s_, o, st = i % len(sets), outs[i % ring], stats[i % ring]
        with_stats = i % 3 != 2
        shards = [x[:M] for x in sets[s_]]
        if with_stats:
            hg.hg_gather_stats(h, shards, [x[:M] for x in o], st[:M], M)
        else:
            hg.hg_gather(h, shards, [x[:M] for x in o], M)
        pend.append((i, s_, M, with_stats))
        if len(pend) == ring or i == n_calls - 1:
            hg.hg_sync(h)
            for j, sj, Mj, ws in pend:
                for d in range(tp):
                    assert torch.equal(outs[j % ring][d][:Mj], want_dev[sj][:Mj]), (j, d, Mj)
                if ws:
                    got = {k: v.cpu().numpy() for k, v in
                           hg.unpack_row_stats(stats[j % ring][:Mj]).items()}
                    for m in range(Mj):
                        mx, arg, se = want_stats[sj][m]
                        assert got["max_logit"][m] == mx and got["argmax"][m] == arg, (j, m)
                        assert abs(got["sum_exp"][m] - se) <= 1e-4 * se, (j, m)
            pend = []
    assert_mailboxes_armed(h, hg)
    h.close()
