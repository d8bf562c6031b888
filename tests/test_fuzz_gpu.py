"""Seeded random configurations of the gather against the CPU oracle.

Each case draws TP in 1..16, an even shard width (so both the 16-byte vector
path and the 4-byte word path occur, with ragged units), a cap, a sequence of
row counts, and a launch shape (elements per lane 1..6, a grid that may be
tiny, prefetch on or off, or the autotuner). Every call is compared with the
oracle word for word; mailboxes and parity are checked after the sequence.
Besides the sentinel and the zero pairs, the inputs carry the generator's
other classes next to the sentinel (swapped zero halves, one-bit neighbours,
NaN and infinity pairs) at 2 %.
"""

import random

import numpy as np
import pytest

import oracle
from tp_vocab_logits_gb300 import hg, synth

from helpers import assert_mailboxes_armed, empty_outs, from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_vocab_logits_gb300 import _build
    _build.build()
    oracle.build()


def draw(case: int) -> dict:
    rng = random.Random(1000 + case)
    tp = rng.choice([1, 2, 3, 4, 5, 7, 8, 11, 16])
    W = 2 * rng.randint(1, 1200) if rng.random() < 0.5 else 8 * rng.randint(1, 400)
    cap = rng.randint(1, 6)
    Ms = [rng.randint(1, cap) for _ in range(rng.randint(2, 5))]
    kw = {}
    if rng.random() < 0.25:
        kw["autotune"] = True
    else:
        if rng.random() < 0.7:
            kw["elems_per_lane"] = rng.randint(1, 6)
        if rng.random() < 0.5:
            kw["ctas"] = rng.choice([1, 2, 3, 5, 17, 64])
        kw["prefetch"] = rng.choice([0, 1, 2])
    return {"tp": tp, "W": W, "cap": cap, "Ms": Ms, "kw": kw}


@pytest.mark.parametrize("case", range(64))
def test_random_configuration_vs_oracle(case):
    c = draw(case)
    tp, W, cap = c["tp"], c["W"], c["cap"]
    h = hg.hg_create(tp, W, cap, **c["kw"])
    og = oracle.Gather(tp, W, cap)
    for i, M in enumerate(c["Ms"]):
        bits = synth.shards(50 + case, tp, M, W, scale=3.0, sent_frac=0.03, zero_frac=0.01,
                            negzero_frac=0.01, extra_frac=0.02,
                            set_index=i).numpy().view(np.uint16)
        want = og.call(bits)
        outs = empty_outs(tp, M, tp * W)
        hg.hg_gather(h, to_dev(bits), outs, M)
        hg.hg_sync(h)
        got = from_dev(outs)
        if not np.array_equal(got, want):
            raise AssertionError(f"{c}: call {i} (M={M}) differs in {int((got != want).sum())} words")
        assert hg.hg_parity(h) == og.parity
    assert_mailboxes_armed(h, hg)
    h.close()


def draw_fused(case: int) -> dict:
    rng = random.Random(5000 + case)
    return {"tp": rng.randint(1, 8), "W": 128 * rng.randint(1, 12), "K": 64 * rng.randint(1, 12),
            "M": rng.randint(1, 16), "ctas": rng.choice([0, 2, 3, 5, 7, 11, 13])}


@pytest.mark.parametrize("case", range(16))
def test_random_fused_configuration(case):
    """The fused LM head + gather on seeded random shapes and grids (tail
    splits of 2..4 parts, unsplit tails, one wave): logits within
    2e-2 + 1e-2 * |ref| of the oracle's float64 product, and the gathered
    outputs bit-exact to hg_gather of those logits."""
    import torch
    c = draw_fused(case)
    tp, W, K, M = c["tp"], c["W"], c["K"], c["M"]
    h = hg.hg_create(tp, W, 16, ctas=c["ctas"])
    weight_cpu = [synth.weight(60 + case, r, W, K) for r in range(tp)]
    hid_cpu = synth.hidden(60 + case, tp, M, K)
    weight = [w.cuda() for w in weight_cpu]
    hidden = [hid_cpu[r].cuda() for r in range(tp)]
    outs = [torch.full((M, tp * W), 0x2222, dtype=torch.int16, device="cuda") for _ in range(tp)]
    logits = [torch.full((M, W), 0x3333, dtype=torch.int16, device="cuda") for _ in range(tp)]
    hg.hg_gather_fused(h, hidden, weight, outs, M, logits=logits)
    hg.hg_sync(h)
    for r in range(tp):
        ref = oracle.lm_head_f64(hid_cpu[r].numpy().view(np.uint16),
                                 weight_cpu[r].numpy().view(np.uint16))
        got = torch.from_numpy(logits[r].cpu().numpy()).view(torch.bfloat16).double().numpy()
        bad = np.abs(got - ref) > 2e-2 + 1e-2 * np.abs(ref)
        assert not bad.any(), f"{c}: rank {r}: {int(bad.sum())} logits outside tolerance"
    h2 = hg.hg_create(tp, W, 16)
    ref_out = [torch.empty_like(o) for o in outs]
    hg.hg_gather(h2, logits, ref_out, M)
    hg.hg_sync(h2)
    h2.close()
    for d in range(tp):
        assert torch.equal(outs[d], ref_out[d]), f"{c}: rank {d} differs from the gather"
    assert_mailboxes_armed(h, hg)
    h.close()
