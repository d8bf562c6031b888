"""Graph-capturable gather: handles created with device_parity keep the parity
in device memory (each reader of a call's kernel reads its own copy of it, and
every copy is flipped once per call after it was read), so calls may be
captured into a CUDA graph and replayed. Parity with the CPU oracle as
everywhere: outputs word for word, mailboxes re-armed, parity sequence."""

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


def test_device_parity_eager_vs_oracle():
    tp, W, cap = 8, 4096, 4
    h = hg.hg_create(tp, W, cap, device_parity=True)
    og = oracle.Gather(tp, W, cap)
    for i, M in enumerate([1, 4, 2, 2, 3, 1]):
        bits = synth.shards(21, tp, M, W, scale=3.0, sent_frac=0.02, set_index=i) \
            .numpy().view(np.uint16)
        want = og.call(bits)
        outs = empty_outs(tp, M, tp * W)
        hg.hg_gather(h, to_dev(bits), outs, M)
        hg.hg_sync(h)
        assert hg.hg_parity(h) == og.parity
        np.testing.assert_array_equal(from_dev(outs), want)
        assert_mailboxes_armed(h, hg)
    h.close()


@pytest.mark.parametrize("tp,W,Ms", [(8, 20480, [1, 2, 1, 8, 3]), (4, 1000, [2, 2, 1])])
def test_graph_capture_replay_vs_oracle(tp, W, Ms):
    cap = max(Ms)
    h = hg.hg_create(tp, W, cap, device_parity=True)
    og = oracle.Gather(tp, W, cap)
    sets = [synth.shards(22, tp, M, W, scale=3.0, sent_frac=0.01, set_index=i)
            .numpy().view(np.uint16) for i, M in enumerate(Ms)]
    dev = [to_dev(b) for b in sets]
    outs = [empty_outs(tp, M, tp * W) for M in Ms]
    # one eager call first (loads the kernels before the capture)
    np.testing.assert_array_equal(og.call(sets[0]), _eager(h, dev[0], outs[0], Ms[0]))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i, M in enumerate(Ms):
            hg.hg_gather(h, dev[i], outs[i], M)
    torch.cuda.synchronize()
    for replay in range(3):
        for o in outs:
            for t in o:
                t.fill_(0x5A5A)
        g.replay()
        torch.cuda.synchronize()
        hg.hg_sync(h)
        for i, M in enumerate(Ms):
            np.testing.assert_array_equal(from_dev(outs[i]), og.call(sets[i]),
                                          err_msg=f"replay {replay} call {i}")
        assert hg.hg_parity(h) == og.parity
        assert_mailboxes_armed(h, hg)
    h.close()


def _eager(h, shards, outs, M):
    hg.hg_gather(h, shards, outs, M)
    hg.hg_sync(h)
    return from_dev(outs)


@pytest.mark.parametrize("ctas", [0, 5])
def test_fused_graph_capture_replay(ctas):
    """The fused LM-head producer on a device-parity handle, captured and
    replayed: outputs equal the unfused gather of its own logits each replay.
    With 5 CTAs the 16 tiles leave one tail tile split into 4 parts, whose
    split cells must be re-armed by every replay."""
    tp, W, K, M = 4, 512, 256, 3
    h = hg.hg_create(tp, W, 4, device_parity=True, ctas=ctas)
    weight = [synth.weight(8, r, W, K, device="cuda") for r in range(tp)]
    hid = synth.hidden(8, tp, M, K, device="cuda")
    hidden = [hid[r] for r in range(tp)]
    outs = [torch.empty((M, tp * W), dtype=torch.int16, device="cuda") for _ in range(tp)]
    logits = [torch.empty((M, W), dtype=torch.int16, device="cuda") for _ in range(tp)]
    hg.hg_gather_fused(h, hidden, weight, outs, M, logits=logits)  # eager first
    hg.hg_sync(h)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hg.hg_gather_fused(h, hidden, weight, outs, M, logits=logits)
        hg.hg_gather_fused(h, hidden, weight, outs, M, logits=logits)
    h2 = hg.hg_create(tp, W, 4)
    for replay in range(2):
        for o in outs:
            o.fill_(7)
        g.replay()
        torch.cuda.synchronize()
        hg.hg_sync(h)
        ref = [torch.empty_like(o) for o in outs]
        hg.hg_gather(h2, logits, ref, M)
        hg.hg_sync(h2)
        for d in range(tp):
            assert torch.equal(outs[d], ref[d]), f"replay {replay} rank {d}"
        assert_mailboxes_armed(h, hg)
    h.close()
    h2.close()


def test_host_buffers_graph_replay_vs_oracle():
    """hg_gather_host on a device-parity handle, captured once (two calls) and
    replayed twice: page-locked host outputs against the oracle run through
    the same four calls."""
    tp, W, cap, M = 4, 1024, 2, 2
    h = hg.hg_create(tp, W, cap, device_parity=True)
    og = oracle.Gather(tp, W, cap)
    sets = [synth.shards(31, tp, M, W, scale=3.0, sent_frac=0.02, set_index=i)
            .numpy().view(np.uint16) for i in range(2)]
    shards = [[torch.from_numpy(b[r].view(np.int16).copy()).pin_memory() for r in range(tp)]
              for b in sets]
    outs = [[torch.zeros((M, tp * W), dtype=torch.int16).pin_memory() for _ in range(tp)]
            for _ in range(2)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(2):
            hg.hg_gather_host(h, shards[i], outs[i], M, stream=s)
    for replay in range(2):
        wants = [og.call(sets[i]) for i in range(2)]
        g.replay()
        torch.cuda.synchronize()
        hg.hg_sync(h)
        for i in range(2):
            got = np.stack([o.numpy().view(np.uint16) for o in outs[i]])
            np.testing.assert_array_equal(got, wants[i], err_msg=f"replay {replay} call {i}")
        assert hg.hg_parity(h) == og.parity
    assert_mailboxes_armed(h, hg)
    h.close()


def test_stats_graph_replay_vs_oracle():
    """hg_gather_stats on a device-parity handle (TP8, V=163840, M=4), two
    calls captured once and replayed twice: outputs and row statistics
    against the oracle each replay (the statistics cells re-arm themselves)."""
    tp, W, cap, M = 8, 20480, 4, 4
    h = hg.hg_create(tp, W, cap, device_parity=True)
    og = oracle.Gather(tp, W, cap)
    sets = [synth.shards(41, tp, M, W, scale=3.0, sent_frac=0.01, set_index=i)
            .numpy().view(np.uint16) for i in range(2)]
    dev = [to_dev(b) for b in sets]
    outs = [empty_outs(tp, M, tp * W) for _ in range(2)]
    stats = [hg.new_row_stats(M) for _ in range(2)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(2):
            hg.hg_gather_stats(h, dev[i], outs[i], stats[i], M, stream=s)
    for replay in range(2):
        wants = [og.call(sets[i]) for i in range(2)]
        g.replay()
        torch.cuda.synchronize()
        hg.hg_sync(h)
        for i in range(2):
            np.testing.assert_array_equal(from_dev(outs[i]), wants[i])
            got = {k: v.cpu().numpy() for k, v in hg.unpack_row_stats(stats[i]).items()}
            for m in range(M):
                mx, arg, se = oracle.row_stats(wants[i][0][m])
                assert got["max_logit"][m] == mx and got["argmax"][m] == arg
                assert abs(got["sum_exp"][m] - se) <= 1e-4 * se
    assert_mailboxes_armed(h, hg)
    h.close()
