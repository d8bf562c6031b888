"""Brute force over the 32-bit word classes next to the sentinel, on the GPU,
against the CPU oracle.

The gather compares every 32-bit word with the sentinel pair (+0, -0) =
0x80000000 twice: once to rewrite a data word equal to it as (+0, +0)
(vLLM API page "...runtime.logits_gather", HeadGather docstring: the bytes
move unchanged but for that pair), and once per poll to decide whether the
word has arrived. A compare that looked at one half of the word only, or at
the sign bits, or that treated a NaN or an infinity specially, would pass
random data and fail on one of these classes:

    0x80000000  the sentinel (+0, -0): sent as (+0, +0)
    0x00000000  (+0, +0)
    0x80008000  (-0, -0)
    0x00008000  (-0, +0), the sentinel's halves swapped
    0x80000001  the sentinel with the lowest bit set
    0x80010000  the sentinel with the lowest bit of the high half set
    0xC0000000  the sentinel with the bit below the sign set
    0x7FC07FC0  a NaN pair
    0xFF80FF80  (-inf, -inf)
    0x7F807F80  (+inf, +inf)
    generic     (1.0 + tiny, ...) words that differ from position to position

At TP=2 every combination of classes over a rank-row pair is issued: on the
4-byte word path (shard width 4, two words per rank-row) all 11^4 = 14641
combinations of the four words of a gathered row, and on the 16-byte vector
path (shard width 8, one vector per rank-row) all 11^4 combinations of the
four words of each rank's vector. They go out as 121 consecutive calls of 121
rows each, over both mailbox parities, and every call's outputs, the parity
and the mailboxes are compared with the oracle run through the same calls.
"""

import numpy as np
import pytest

import oracle
from tp_vocab_logits_gb300 import hg

from helpers import empty_outs, from_dev, to_dev

SPECIAL = [0x80000000, 0x00000000, 0x80008000, 0x00008000, 0x80000001, 0x80010000,
           0xC0000000, 0x7FC07FC0, 0xFF80FF80, 0x7F807F80]
N_CLASSES = len(SPECIAL) + 1  # the last class is a generic data word
N = N_CLASSES * N_CLASSES     # class pairs: calls, and rows per call


@pytest.fixture(scope="module")
def _built():
    from tp_vocab_logits_gb300 import _build
    _build.build()
    oracle.build()


def classify(w: int) -> int:
    """Class index of a word built by `word`."""
    return SPECIAL.index(w) if w in SPECIAL else len(SPECIAL)


def word(cls: int, rank: int, call: int, row: int, pos: int) -> int:
    """The word of class `cls`; the generic class is 1.0 in the high half and
    a low half that depends on where the word sits, so a word moved to the
    wrong place is seen."""
    if cls < len(SPECIAL):
        return SPECIAL[cls]
    return 0x3F800000 | ((rank * 4099 + call * 131 + row * 17 + pos * 5) & 0x7FFF)


def call_words(call: int, words_per_rank: int) -> np.ndarray:
    """[2, N, words_per_rank] uint32 shards of call `call` (rows = class pairs).

    Word path (2 words per rank-row): rank 0's words are the call's class
    pair, rank 1's the row's class pair, so the four words of a gathered row
    run over every combination in the 121 calls. Vector path (4 words per
    rank-row): rank 0's vector is (call pair, row pair) and rank 1's (row
    pair, call pair), so each rank's vector runs over every combination."""
    out = np.empty((2, N, words_per_rank), dtype=np.uint32)
    ca, cb = divmod(call, N_CLASSES)
    for m in range(N):
        ma, mb = divmod(m, N_CLASSES)
        if words_per_rank == 2:
            cls = [[ca, cb], [ma, mb]]
        else:
            cls = [[ca, cb, ma, mb], [ma, mb, ca, cb]]
        for r in range(2):
            for k in range(words_per_rank):
                out[r, m, k] = word(cls[r][k], r, call, m, k)
    return out


def test_calls_cover_every_class_combination():
    """The 121 calls issue every combination of the 11 classes over the four
    words of a gathered row (word path) and over the four words of each rank's
    vector (vector path)."""
    rows2, vec0, vec1 = set(), set(), set()
    for call in range(N):
        w2 = call_words(call, 2)
        w4 = call_words(call, 4)
        for m in range(N):
            rows2.add(tuple(classify(int(x)) for x in np.concatenate([w2[0, m], w2[1, m]])))
            vec0.add(tuple(classify(int(x)) for x in w4[0, m]))
            vec1.add(tuple(classify(int(x)) for x in w4[1, m]))
    assert len(rows2) == len(vec0) == len(vec1) == N_CLASSES ** 4


@pytest.mark.gpu
@pytest.mark.parametrize("W,kw", [
    (4, {}),                                                # word path, fixed launch rule
    (8, {}),                                                # vector path, fixed launch rule
    (8, {"elems_per_lane": 1, "ctas": 3, "prefetch": 1}),   # few CTAs looping over units
    (4, {"elems_per_lane": 2, "ctas": 5}),
    (8, {"device_parity": True}),                           # parity read from device memory
])
def test_word_classes_brute_force(_built, W, kw):
    tp = 2
    wpr = W // 2
    h = hg.hg_create(tp, W, N, **kw)
    og = oracle.Gather(tp, W, N)
    for call in range(N):
        words = call_words(call, wpr)
        bits = words.view(np.uint16).reshape(tp, N, W)
        want = og.call(bits)
        outs = empty_outs(tp, N, tp * W)
        hg.hg_gather(h, to_dev(bits), outs, N)
        hg.hg_sync(h)
        got = from_dev(outs)
        if not np.array_equal(got, want):
            gw = got.view(np.uint32)
            ww = want.view(np.uint32)
            bad = np.argwhere(gw != ww)
            d, m, k = bad[0]
            raise AssertionError(f"call {call}: {len(bad)} words differ; first at rank {d} row "
                                 f"{m} word {k}: got {gw[d, m, k]:#010x}, want {ww[d, m, k]:#010x}")
        assert hg.hg_parity(h) == og.parity
        if call % 20 == 0 or call == N - 1:
            for d in range(tp):
                mb = hg.mailbox_words(h, d).cpu().numpy().view(np.uint32)
                for q in range(2):
                    np.testing.assert_array_equal(mb[q], og.mailbox(d, q))
    h.close()


def test_every_class_moves_unchanged_but_the_sentinel():
    """The oracle's expectation itself, per class, on the vector path: every
    class but the sentinel comes out as it went in, the sentinel as zero (so a
    pass above cannot come from an oracle that moves everything unchanged)."""
    oracle.build()
    words = call_words(0, 4)
    og = oracle.Gather(2, 8, N)
    out = og.call(words.view(np.uint16).reshape(2, N, 8)).view(np.uint32)
    concat = np.concatenate([words[0], words[1]], axis=1)
    expect = np.where(concat == 0x80000000, 0, concat).astype(np.uint32)
    np.testing.assert_array_equal(out[0], expect)
    assert (concat == 0x80000000).any()
