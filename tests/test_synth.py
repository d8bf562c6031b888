"""The seeded input generator, on the CPU: its finaliser against splitmix64's
published outputs, and the property the tests rely on, that a value depends
only on its indices (any slice regenerates alone; the shape of the request
changes nothing), plus the injected word classes and the padded-vocab pads."""

import numpy as np
import torch

from tp_vocab_logits_gb300 import synth

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def test_finaliser_matches_splitmix64_from_seed_zero():
    """splitmix64 from state 0 adds the golden gamma and finalises: its first
    outputs are the published 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
    0x06C45D188009454F, 0xF88BB8A8724C81EC, 0x1B39896A51A8749B."""
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
            0xF88BB8A8724C81EC, 0x1B39896A51A8749B]
    got = [synth._mix_int((k * GAMMA) & M64) for k in range(1, 6)]
    assert got == want
    # the tensor form agrees with the integer form (two's-complement int64)
    z = torch.tensor([((k * GAMMA) & M64) - (1 << 64) if ((k * GAMMA) & M64) >= (1 << 63)
                      else (k * GAMMA) & M64 for k in range(1, 6)], dtype=torch.int64)
    t = [int(v) & M64 for v in synth._mix(z).tolist()]
    assert t == want


def test_shard_values_depend_only_on_their_indices():
    full = synth.shards(7, 4, 6, 64, scale=3.0, sent_frac=0.05, zero_frac=0.02,
                        negzero_frac=0.02, set_index=3)
    part = synth.shards(7, 2, 3, 16, scale=3.0, sent_frac=0.05, zero_frac=0.02,
                        negzero_frac=0.02, set_index=3, rank0=1, row0=2, col0=32)
    assert torch.equal(part, full[1:3, 2:5, 32:48])
    # fewer rows requested: the rows that are generated are the same
    assert torch.equal(synth.shards(7, 4, 2, 64, scale=3.0, set_index=3),
                       synth.shards(7, 4, 6, 64, scale=3.0, set_index=3)[:, :2])
    # another set or seed gives other values
    assert not torch.equal(synth.shards(7, 4, 6, 64, set_index=4),
                           synth.shards(7, 4, 6, 64, set_index=3))
    assert not torch.equal(synth.shards(8, 4, 6, 64, set_index=3),
                           synth.shards(7, 4, 6, 64, set_index=3))


def test_weight_blocks_regenerate_alone():
    w = synth.weight(4, 3, 256, 96)
    assert torch.equal(synth.weight(4, 3, 64, 96, row0=128), w[128:192])
    assert not torch.equal(synth.weight(4, 2, 256, 96), w)


def test_injected_word_classes_and_pads():
    s = synth.shards(11, 2, 8, 4096, scale=2.0, sent_frac=0.1, zero_frac=0.05,
                     negzero_frac=0.05).numpy().view(np.uint32)
    n = s.size
    for word, p in ((0x80000000, 0.1), (0x00000000, 0.05), (0x80008000, 0.05)):
        frac = np.count_nonzero(s == word) / n
        assert abs(frac - p) < 0.01, (hex(word), frac)
    bits = synth.shards(11, 4, 2, 16, v_real=4 * 16 - 3).numpy().view(np.uint16)
    assert (bits[3, :, 13:] == 0xFF80).all()            # the last 3 columns of the row
    assert not (bits[3, :, :13] == 0xFF80).any() and not (bits[:3] == 0xFF80).any()


def test_normal_values_have_the_requested_spread():
    v = synth.shards(5, 8, 4, 4096, scale=3.0).view(torch.bfloat16).float()
    assert abs(v.mean().item()) < 0.05 and abs(v.std().item() - 3.0) < 0.05
    u = synth.shards(5, 8, 4, 4096, dist="uniform", scale=20.0).view(torch.bfloat16).float()
    assert u.min().item() >= -20.0 and u.max().item() <= 20.0
    assert abs(u.std().item() - 20.0 / 3 ** 0.5) < 0.2


def test_extra_word_classes():
    """extra_frac injects each word of EXTRA_WORDS at an equal share, leaves
    the other words as they were, and with 0 changes nothing."""
    kw = dict(scale=2.0, sent_frac=0.02, zero_frac=0.01, negzero_frac=0.01, set_index=2)
    base = synth.shards(13, 2, 8, 4096, **kw)
    assert torch.equal(synth.shards(13, 2, 8, 4096, extra_frac=0.0, **kw), base)
    ex = synth.shards(13, 2, 8, 4096, extra_frac=0.14, **kw)
    b = base.numpy().view(np.uint32)
    e = ex.numpy().view(np.uint32)
    changed = b != e
    n = e.size
    assert abs(np.count_nonzero(changed) / n - 0.14) < 0.01
    for word in synth.EXTRA_WORDS:
        assert word != 0x80000000
        frac = np.count_nonzero(e[changed] == word) / n
        assert abs(frac - 0.02) < 0.004, (hex(word), frac)
    assert set(np.unique(e[changed]).tolist()) <= set(synth.EXTRA_WORDS)
    # slices regenerate alone with the extra classes too
    part = synth.shards(13, 1, 3, 16, extra_frac=0.14, rank0=1, row0=2, col0=32, **kw)
    assert torch.equal(part, ex[1:2, 2:5, 32:48])
