"""The drafter's gather beside the target's, on one stream.

The vLLM API page "...runtime.logits_gather" (module docstring) says the
target's gather runs as the DSpark drafter's logits gather does: the same
kernel and the same mailbox class, with the drafter's own shapes. So a decode
step issues two gathers of two handles back to back on one stream: the
drafter's, over its block of draft positions, then the target's, which
verifies the token before them plus the drafted ones. The pages give no
drafter shape; the reading used here is a drafter with the target's tokenizer
and tensor-parallel group (TP8, V=163840) that drafts a block of 1..4
positions per step (rows {1, 2, 3, 4}), and a target with rows
{1, 2, 3, 4, 5, 8} that gathers 1 + (drafted rows) per step.

Consecutive launches of different handles overlap exactly as those of one
handle do (a programmatic dependent launch: the next kernel starts while the
previous one runs and waits for it before touching memory). Every call of
each handle is compared with its own oracle instance, word for word, with
the parities and mailboxes of both handles checked too.
"""

import numpy as np
import pytest
import torch

import oracle
from tp_vocab_logits_gb300 import hg, synth

from helpers import assert_mailboxes_armed, empty_outs, from_dev, to_dev

pytestmark = pytest.mark.gpu

TP, W = 8, 20480
V = TP * W
DRAFT_ROWS = [1, 2, 3, 4]
TARGET_ROWS = [1, 2, 3, 4, 5, 8]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_vocab_logits_gb300 import _build
    _build.build()
    oracle.build()


def step_inputs(seed, steps):
    """Per step: (drafter rows, drafter shards, target rows, target shards) as
    uint16 bit arrays; the drafter's rows follow a seeded sequence."""
    md = synth.row_sequence(seed, steps, DRAFT_ROWS)
    out = []
    for i, m in enumerate(md):
        d = synth.shards(seed, TP, m, W, scale=3.0, sent_frac=0.01, extra_frac=0.002,
                         set_index=2 * i).numpy().view(np.uint16)
        t = synth.shards(seed + 1, TP, 1 + m, W, scale=3.0, sent_frac=0.01, extra_frac=0.002,
                         set_index=2 * i + 1).numpy().view(np.uint16)
        out.append((m, d, 1 + m, t))
    return out


@pytest.mark.parametrize("device_parity", [False, True])
def test_drafter_and_target_interleaved_eager(device_parity):
    """60 steps issued back to back with no synchronisation between them; all
    checked at the end against two oracle instances."""
    hd = hg.hg_create(TP, W, max(DRAFT_ROWS), DRAFT_ROWS, device_parity=device_parity)
    ht = hg.hg_create(TP, W, 8, TARGET_ROWS, device_parity=device_parity)
    od = oracle.Gather(TP, W, max(DRAFT_ROWS), DRAFT_ROWS)
    ot = oracle.Gather(TP, W, 8, TARGET_ROWS)
    steps = step_inputs(31 + device_parity, 60)
    issued = []
    for md, d, mt, t in steps:
        outs_d = empty_outs(TP, md, V)
        outs_t = empty_outs(TP, mt, V)
        hg.hg_gather(hd, to_dev(d), outs_d, md)
        hg.hg_gather(ht, to_dev(t), outs_t, mt)
        issued.append((outs_d, outs_t))
    hg.hg_sync(hd)
    hg.hg_sync(ht)
    for i, ((md, d, mt, t), (outs_d, outs_t)) in enumerate(zip(steps, issued)):
        np.testing.assert_array_equal(from_dev(outs_d), od.call(d), err_msg=f"step {i} drafter")
        np.testing.assert_array_equal(from_dev(outs_t), ot.call(t), err_msg=f"step {i} target")
    assert hg.hg_parity(hd) == od.parity and hg.hg_parity(ht) == ot.parity
    assert_mailboxes_armed(hd, hg)
    assert_mailboxes_armed(ht, hg)
    hd.close()
    ht.close()


def test_drafter_and_target_interleaved_graph_replay():
    """A CUDA graph of 24 captured steps (drafter then target, 48 launches),
    replayed 4 times back to back; after every replay every call's outputs
    against the two oracles, which run through the same calls in the same
    order, and both handles' parities and mailboxes."""
    hd = hg.hg_create(TP, W, max(DRAFT_ROWS), DRAFT_ROWS, device_parity=True)
    ht = hg.hg_create(TP, W, 8, TARGET_ROWS, device_parity=True)
    od = oracle.Gather(TP, W, max(DRAFT_ROWS), DRAFT_ROWS)
    ot = oracle.Gather(TP, W, 8, TARGET_ROWS)
    steps = step_inputs(41, 24)
    dev = [(to_dev(d), to_dev(t)) for _, d, _, t in steps]
    outs = [(empty_outs(TP, md, V), empty_outs(TP, mt, V)) for md, _, mt, _ in steps]
    # one eager step first (loads the kernels before the capture)
    md0, d0, mt0, t0 = steps[0]
    hg.hg_gather(hd, dev[0][0], outs[0][0], md0)
    hg.hg_gather(ht, dev[0][1], outs[0][1], mt0)
    hg.hg_sync(hd)
    hg.hg_sync(ht)
    np.testing.assert_array_equal(from_dev(outs[0][0]), od.call(d0))
    np.testing.assert_array_equal(from_dev(outs[0][1]), ot.call(t0))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for (md, _, mt, _), (sd, st), (o_d, o_t) in zip(steps, dev, outs):
            hg.hg_gather(hd, sd, o_d, md)
            hg.hg_gather(ht, st, o_t, mt)
    torch.cuda.synchronize()
    for replay in range(4):
        for o_d, o_t in outs:
            for x in o_d + o_t:
                x.fill_(0x5A5A)
        g.replay()
        torch.cuda.synchronize()
        hg.hg_sync(hd)
        hg.hg_sync(ht)
        for i, ((md, d, mt, t), (o_d, o_t)) in enumerate(zip(steps, outs)):
            np.testing.assert_array_equal(from_dev(o_d), od.call(d),
                                          err_msg=f"replay {replay} step {i} drafter")
            np.testing.assert_array_equal(from_dev(o_t), ot.call(t),
                                          err_msg=f"replay {replay} step {i} target")
        assert hg.hg_parity(hd) == od.parity and hg.hg_parity(ht) == ot.parity
        assert_mailboxes_armed(hd, hg)
        assert_mailboxes_armed(ht, hg)
    del g
    hd.close()
    ht.close()
