"""The measurement surface of the library on the GPU: the timeline build of
the gather (per-CTA %globaltimer records) and the latency-floor kernels.

The timeline build must change no result (outputs against the oracle), and
its records must follow the launch semantics: within a CTA, entry <= end of
the wait <= each warp's end; and across consecutive calls on one stream, a
call's wait returns only after the previous call's kernel completed, so no
CTA of call i+1 passes its wait before every warp of call i has finished
(the programmatic dependent launch lets call i+1 start early, but not touch
memory early). The handoff floor kernel must hand every CTA's token to its
neighbour and leave its slots re-armed.
"""

import numpy as np
import pytest
import torch

import oracle
from tp_vocab_logits_gb300 import hg, synth

from helpers import assert_mailboxes_armed, empty_outs, from_dev, to_dev

pytestmark = pytest.mark.gpu
S_U32 = 0x80000000


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_vocab_logits_gb300 import _build
    _build.build()
    oracle.build()


@pytest.mark.parametrize("stats", [False, True])
def test_timeline_records_follow_the_launch_order(stats):
    tp, W, cap, n = 8, 20480, 8, 12
    h = hg.hg_create(tp, W, cap, timeline_calls=n)
    og = oracle.Gather(tp, W, cap)
    Ms = [1, 8, 1, 4, 2, 8, 1, 1, 3, 8, 5, 1]
    wants, outs_all, grids = [], [], []
    st = hg.new_row_stats(cap)
    for i, M in enumerate(Ms):
        bits = synth.shards(71, tp, M, W, scale=3.0, sent_frac=0.01, set_index=i) \
            .numpy().view(np.uint16)
        wants.append(og.call(bits))
        outs = empty_outs(tp, M, tp * W)
        if stats:
            hg.hg_gather_stats(h, to_dev(bits), outs, st[:M], M)
        else:
            hg.hg_gather(h, to_dev(bits), outs, M)
        outs_all.append(outs)
        grids.append(hg.hg_launch_shape(h, M)["ctas"] if not stats else None)
    hg.hg_sync(h)
    for i, (want, outs) in enumerate(zip(wants, outs_all)):
        np.testing.assert_array_equal(from_dev(outs), want, err_msg=f"call {i}")
    assert_mailboxes_armed(h, hg)
    rec, nxt = hg.hg_timeline(h)
    assert nxt == len(Ms) % n
    rec = rec.cpu().numpy()
    prev_end = None
    # the last n calls, in call order
    order = [(nxt + k) % n for k in range(n)]
    for k, slot in enumerate(order):
        i = len(Ms) - n + k
        r = rec[slot]
        used = r[:, 0] > 0
        grid = int(used.sum())
        if grids[i] is not None:
            assert grid >= grids[i], f"call {i}: {grid} CTAs recorded, grid {grids[i]}"
        r = r[used]
        ends = r[:, 2:2 + tp]
        assert (ends > 0).all(), f"call {i}: a warp recorded no end"
        assert (r[:, 0] <= r[:, 1]).all() and (r[:, 1:2] <= ends).all()
        if prev_end is not None:
            # 64 ns of slack for the timer's granularity
            assert r[:, 1].min() + 64 >= prev_end, f"call {i} passed its wait early"
        prev_end = ends.max()
    h.close()


def test_timeline_needs_the_vector_path():
    with pytest.raises(hg.HGError) as e:
        hg.hg_create(2, 6, 2, timeline_calls=4)          # word path
    assert e.value.status == hg.HG_ERR_ARG
    with pytest.raises(hg.HGError) as e:
        hg.hg_create(2, 64, 2, timeline_calls=4, prefetch=1)
    assert e.value.status == hg.HG_ERR_ARG
    h = hg.hg_create(2, 64, 2)
    with pytest.raises(hg.HGError):
        hg.hg_timeline(h)                                 # no timeline
    h.close()


@pytest.mark.parametrize("ctas,threads", [(216, 256), (608, 256), (5, 32)])
def test_handoff_probe_hands_every_token_to_its_neighbour(ctas, threads):
    nbytes = hg.hg_probe_scratch_bytes(ctas, threads)
    scratch = torch.zeros(nbytes // 4, dtype=torch.int32, device="cuda")
    hg.hg_probe(2, ctas, threads, scratch)
    for _ in range(3):
        hg.hg_probe(1, ctas, threads, scratch)
        hg.hg_probe(0, ctas, threads)
    torch.cuda.synchronize()
    n = ctas * threads
    words = scratch.cpu().numpy().view(np.uint32)
    slots = words[:4 * n].reshape(ctas, threads, 4)
    outs = words[4 * n:8 * n].reshape(ctas, threads, 4)
    status = int(words[8 * n])
    assert status == 0
    assert (slots == S_U32).all()
    cons = (np.arange(ctas) + 1) % ctas
    np.testing.assert_array_equal(outs[:, :, 0], np.broadcast_to(cons[:, None], (ctas, threads)))
    np.testing.assert_array_equal(outs[:, :, 1], np.broadcast_to(np.arange(threads), (ctas, threads)))
    assert (outs[:, :, 2] == 1).all() and (outs[:, :, 3] == 2).all()


def test_probe_refuses_a_grid_that_cannot_be_resident():
    big = 152 * 64 + 1
    scratch = torch.zeros(hg.hg_probe_scratch_bytes(big, 512) // 4, dtype=torch.int32,
                          device="cuda")
    with pytest.raises(hg.HGError) as e:
        hg.hg_probe(1, big, 512, scratch)
    assert e.value.status == hg.HG_ERR_ARG
