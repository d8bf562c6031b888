"""Sampler statistics folded into the gather's pollers (hg_gather_stats).

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
