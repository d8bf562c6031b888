"""Pins of the CPU oracle against what the pages and the mathematics fix.

The gather's definition comes from the vLLM API page
"vllm.models.kimi_k3.nvidia.specialized_decode.runtime.logits_gather" (module
docstring; class HeadGather: docstring, __init__, __call__) and the pull
request "[Perf][Kimi-K3] Use the one-shot custom all-gather for TP logits"
("Purpose": rank-order concat, padded-vocab slice). The pages print no worked
numbers, so the oracle is pinned by:
  * a hand-worked example (tests/golden/worked_tp2_w4.json);
  * the sentinel's encoding, derived here from torch's own bf16 encoding;
  * invariants I1-I7: concat equality without sentinels (against numpy's
    concatenate), exact sentinel positions, re-armed mailboxes, the parity
    sequence and rejected calls, identical outputs on every rank, an
    exhaustive brute force at TP=2, V=8, and the padded-vocab slice;
  * for the LM head: one-hot closed forms, K=1, and numpy's float64 matmul;
  * for the row statistics: numpy/scipy, closed forms and a hand-worked row.
Every check runs against the real oracle and against mutants of it with a
planted mistake (compiled from a patched copy of the source); each mutant must
fail at least one check.
"""

import itertools
import json
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tp_vocab_logits_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
S = 0x80000000


def _words(bits_u16):
    return np.ascontiguousarray(bits_u16).view(np.uint32)


def _bits_from_words(words_u32):
    return np.ascontiguousarray(np.asarray(words_u32, dtype=np.uint32)).view(np.uint16)


def _rand_words(rng, shape, s_frac=0.0):
    w = rng.integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32)
    w[w == S] = 1
    if s_frac:
        w[rng.random(shape) < s_frac] = S
    return w


# ----------------------------------------------------------------- checks --

def check_sentinel(lib):
    """The sentinel is the BF16 pair (+0, -0) (module docstring): element 2k
    is +0, element 2k+1 is -0, seen as one little-endian 32-bit word."""
    pair = torch.tensor([0.0, -0.0], dtype=torch.bfloat16).view(torch.int32).item() & 0xFFFFFFFF
    assert oracle.sentinel(lib) == pair == S


def check_worked_example(lib):
    with open(os.path.join(HERE, "golden", "worked_tp2_w4.json")) as f:
        ex = json.load(f)
    g = oracle.Gather(ex["tp"], ex["shard_cols"], ex["cap"], ex["rows"], lib=lib)
    for c in ex["calls"]:
        assert g.parity == c["parity_before"]
        shards = np.array([[[int(x, 16) for x in row] for row in r] for r in c["shards"]],
                          dtype=np.uint32)
        st, out = g.call_status(_bits_from_words(shards))
        assert st == c["status"]
        if st == 0:
            want = np.array([[int(x, 16) for x in row] for row in c["out"]], dtype=np.uint32)
            for d in range(ex["tp"]):
                np.testing.assert_array_equal(_words(out[d]), want)
        assert g.parity == c["parity_after"]
        for d in range(ex["tp"]):
            for q in range(2):
                assert (g.mailbox(d, q) == S).all()


def check_config1_golden(lib):
    with open(os.path.join(HERE, "golden", "config1_tiny.json")) as f:
        gd = json.load(f)
    g = oracle.Gather(gd["tp"], gd["shard_cols"], gd["cap"], lib=lib)
    for c in gd["calls"]:
        shards = np.array([[[int(x, 16) for x in row] for row in r] for r in c["shards"]],
                          dtype=np.uint32)
        assert g.parity == c["parity_before"]
        out = g.call(_bits_from_words(shards))
        want = np.array([[[int(x, 16) for x in row] for row in r] for r in c["out"]],
                        dtype=np.uint32)
        np.testing.assert_array_equal(_words(out), want)
        assert g.parity == c["parity_after"]


def check_concat_without_sentinels(lib):
    """I1: with no sentinel word in the input, every output is the rank-order
    concat of the shards (NCCL all-gather layout, module docstring)."""
    rng = np.random.default_rng(11)
    for tp, W, cap in [(2, 8, 3), (3, 6, 2), (4, 64, 5), (8, 16, 8)]:
        g = oracle.Gather(tp, W, cap, lib=lib)
        for M in [1, cap, max(1, cap - 1), 1]:
            sh = _bits_from_words(_rand_words(rng, (tp, M, W // 2))).reshape(tp, M, W)
            out = g.call(sh)
            cat = np.concatenate([sh[r] for r in range(tp)], axis=1)
            for d in range(tp):
                np.testing.assert_array_equal(out[d], cat)


def check_sentinel_positions(lib):
    """I2: with sentinel words injected, the output differs from the concat at
    exactly those words, and holds (+0, +0) there; no output word is the
    sentinel."""
    rng = np.random.default_rng(12)
    tp, W, cap = 4, 32, 4
    g = oracle.Gather(tp, W, cap, lib=lib)
    for M in [4, 2, 3, 1]:
        wd = _rand_words(rng, (tp, M, W // 2), s_frac=0.2)
        wd[0, 0, 0] = S
        out = _words(g.call(_bits_from_words(wd).reshape(tp, M, W)))
        cat = np.concatenate([wd[r] for r in range(tp)], axis=1)
        diff = out[0] != cat
        np.testing.assert_array_equal(diff, cat == S)
        assert diff.sum() == (wd == S).sum() > 0
        assert (out[0][diff] == 0).all()
        assert not (out == S).any()


def check_rearm_and_parity(lib):
    """I3/I4: after each served call every word of every mailbox (both
    parities) is the sentinel again and the parity alternates 0, 1, 0, ...;
    calls whose row count is not served change neither (HeadGather.__call__
    returns before `self.parity ^= 1`)."""
    rng = np.random.default_rng(13)
    tp, W, cap = 3, 10, 4
    g = oracle.Gather(tp, W, cap, rows=[1, 3], lib=lib)
    seq = []
    for M in [1, 3, 2, 0, 5, 3, 1, 4, 1]:
        before = g.parity
        st, _ = g.call_status(_bits_from_words(_rand_words(rng, (tp, max(M, 1), W // 2)))
                              .reshape(tp, max(M, 1), W)[:, :M] if M else
                              np.zeros((tp, 0, W), dtype=np.uint16))
        if M in (1, 3):
            assert st == 0
            seq.append(before)
            assert g.parity == before ^ 1
        else:
            assert st == -1
            assert g.parity == before
        for d in range(tp):
            for q in range(2):
                assert (g.mailbox(d, q) == S).all()
    assert seq == [0, 1, 0, 1, 0]


def check_identical_outputs(lib):
    """I5: every rank's mailbox receives every shard, so all outputs agree."""
    rng = np.random.default_rng(14)
    tp, W = 5, 12
    g = oracle.Gather(tp, W, 2, lib=lib)
    out = _words(g.call(_bits_from_words(_rand_words(rng, (tp, 2, W // 2), 0.3))
                        .reshape(tp, 2, W)))
    for d in range(1, tp):
        np.testing.assert_array_equal(out[d], out[0])


def check_brute_force_tp2_v8(lib):
    """I6: TP=2, V=8 (4 words), every word over {S, (+0,+0), (-0,-0),
    (-0,+0), a generic word}: 625 inputs as consecutive calls, each against
    the definition written independently here."""
    vals = [S, 0x00000000, 0x80008000, 0x00008000, 0x3F80C0A0]
    g = oracle.Gather(2, 4, 1, lib=lib)
    for i, combo in enumerate(itertools.product(vals, repeat=4)):
        wd = np.array(combo, dtype=np.uint32).reshape(2, 1, 2)
        out = _words(g.call(_bits_from_words(wd).reshape(2, 1, 4)))
        want = [0 if x == S else x for x in combo]
        assert out.tolist() == [[want], [want]]
        assert g.parity == (i + 1) % 2
    for d in range(2):
        for q in range(2):
            assert (g.mailbox(d, q) == S).all()


def check_slice(lib):
    """I7: the padded-vocab slice keeps the first v_real bf16 columns; the pad
    columns of the unsliced output hold bf16 -inf."""
    tp, W, M, v_real = 4, 6, 2, 21
    sh = synth.shards(2, tp, M, W, v_real=v_real, scale=3.0).numpy().view(np.uint16)
    g = oracle.Gather(tp, W, M, lib=lib)
    out = g.call(sh)
    full = np.concatenate([sh[r] for r in range(tp)], axis=1)
    assert (out[0][:, v_real:] == 0xFF80).all()
    sl = oracle.slice_vocab(out[1], v_real, lib=lib)
    assert sl.shape == (M, v_real)
    np.testing.assert_array_equal(sl, full[:, :v_real])


def _bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _bf16_vals(bits):
    return torch.tensor(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def check_lm_head_one_hot(lib):
    """logits[m][n] = sum_k hidden[m][k] * weight[n][k]: a one-hot hidden row
    at k0 picks weight[:, k0] exactly; K=1 is a plain product."""
    rng = np.random.default_rng(15)
    M, K, W = 3, 9, 7
    wt = _bf16_bits(rng.standard_normal((W, K)))
    h = np.zeros((M, K), dtype=np.float32)
    ks = [0, 4, 8]
    for m, k0 in enumerate(ks):
        h[m, k0] = 1.0
    out = oracle.lm_head_f64(_bf16_bits(h), wt, lib=lib)
    wv = _bf16_vals(wt)
    for m, k0 in enumerate(ks):
        np.testing.assert_array_equal(out[m], wv[:, k0])
    h1 = _bf16_bits(rng.standard_normal((2, 1)))
    w1 = _bf16_bits(rng.standard_normal((5, 1)))
    out1 = oracle.lm_head_f64(h1, w1, lib=lib)
    np.testing.assert_array_equal(out1, np.outer(_bf16_vals(h1)[:, 0], _bf16_vals(w1)[:, 0]))


def check_lm_head_matmul(lib):
    """Non-square random case against numpy's float64 matmul (hidden @
    weight.T), and a column range against the same columns of the full call."""
    rng = np.random.default_rng(16)
    M, K, W = 5, 37, 23
    h = _bf16_bits(rng.standard_normal((M, K)))
    wt = _bf16_bits(rng.standard_normal((W, K)) * 0.02)
    out = oracle.lm_head_f64(h, wt, lib=lib)
    ref = _bf16_vals(h) @ _bf16_vals(wt).T
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
    part = oracle.lm_head_f64(h, wt, 5, 17, lib=lib)
    np.testing.assert_array_equal(part, out[:, 5:17])


def check_row_stats(lib):
    """Sampler statistics: against numpy/scipy on random rows (max, first
    argmax, logsumexp), closed forms (a constant row: sum_exp = V, argmax 0),
    ties resolved to the smallest index, -inf pads excluded from the sum, and
    a hand-worked row."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(17)
    for V in (1, 7, 64, 1000):
        bits = _bf16_bits(rng.standard_normal(V) * 3)
        vals = _bf16_vals(bits)
        mx, arg, se = oracle.row_stats(bits, lib=lib)
        assert mx == vals.max() and arg == int(np.argmax(vals))
        np.testing.assert_allclose(mx + np.log(se), logsumexp(vals), rtol=1e-13, atol=1e-13)
    mx, arg, se = oracle.row_stats(_bf16_bits(np.full(50, 1.5)), lib=lib)
    assert (mx, arg, se) == (1.5, 0, 50.0)
    assert oracle.row_stats(_bf16_bits(np.array([0.0, 2.0, -1.0, 2.0])), lib=lib)[1] == 1
    # hand-worked: [0.69140625, -inf, +0]: max at 0, sum = 1 + exp(-0.69140625)
    mx, arg, se = oracle.row_stats(np.array([0x3F31, 0xFF80, 0x0000], dtype=np.uint16), lib=lib)
    assert mx == 0.69140625 and arg == 0
    assert abs(se - (1.0 + np.exp(-0.69140625))) < 1e-15
    mx, arg, se = oracle.row_stats(np.array([0xFF80, 0xFF80], dtype=np.uint16), lib=lib)
    assert mx == -np.inf and arg == 0 and se == 0.0


CHECKS = [check_sentinel, check_worked_example, check_config1_golden,
          check_concat_without_sentinels, check_sentinel_positions, check_rearm_and_parity,
          check_identical_outputs, check_brute_force_tp2_v8, check_slice,
          check_lm_head_one_hot, check_lm_head_matmul, check_row_stats]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_mod, check):
    check(oracle_mod.load())


def test_config1_inputs_regenerate():
    """The stored config-1 inputs are what the seeded generator makes."""
    with open(os.path.join(HERE, "golden", "config1_tiny.json")) as f:
        gd = json.load(f)
    for i, c in enumerate(gd["calls"]):
        s = synth.shards(0, gd["tp"], 1, gd["shard_cols"], sent_frac=0.02, zero_frac=0.01,
                         negzero_frac=0.01, set_index=i).numpy().view(np.uint16)
        want = np.array([[[int(x, 16) for x in row] for row in r] for r in c["shards"]],
                        dtype=np.uint32)
        np.testing.assert_array_equal(_words(s), want)


# ------------------------------------------------------------------ mutants --
# Each entry plants one plausible mistake in a copy of the oracle's source.
MUTANTS = {
    "no_rewrite": ("(x == kSentinel) ? kSentinelSentAs : x", "x"),
    "wrong_rewrite_value": ("pair_word(kBf16PosZero, kBf16PosZero)",
                            "pair_word(kBf16NegZero, kBf16PosZero)"),
    "swapped_sentinel_halves": ("pair_word(kBf16PosZero, kBf16NegZero)",
                                "pair_word(kBf16NegZero, kBf16PosZero)"),
    "wrong_rank_offset": ("g->at(d, q, m, r * w + j)", "g->at(d, q, m, j * tp + r)"),
    "push_own_rank_only": ("for (int d = 0; d < tp; ++d) g->box[g->at(d, q, m, r * w + j)] = y;",
                           "g->box[g->at(r, q, m, r * w + j)] = y;"),
    "no_rearm": ("g->box[g->at(d, q, m, k)] = kSentinel;\n", "\n"),
    "no_parity_flip": ("g->parity ^= 1;", ";"),
    "serves_unlisted_rows": ("if (M < 1 || M > g->cap || !g->served[M]) return -1;",
                             "if (M < 1 || M > g->cap) return -1;"),
    "rows_from_wrong_rank": ("shard[((size_t)r * M + m) * w + j]",
                             "shard[((size_t)((r + 1) % tp) * M + m) * w + j]"),
    "lm_head_transposed_hidden": ("hidden[(size_t)m * K + k]", "hidden[(size_t)k * M + m]"),
    "lm_head_dropped_term": ("for (int k = 0; k < K; ++k)", "for (int k = 1; k < K; ++k)"),
    "bf16_widening_shift": ("(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    "slice_wrong_stride": ("out[(size_t)m * V + c]", "out[(size_t)m * v_real + c]"),
    "stats_last_argmax": ("if (x > mx) { mx = x; arg = c; }", "if (x >= mx) { mx = x; arg = c; }"),
    "stats_sum_without_shift": ("s += std::exp(x - mx);", "s += std::exp(x);"),
    "stats_sum_unguarded": ("if (x != -std::numeric_limits<double>::infinity()) s += std::exp(x - mx);",
                            "s += std::exp(x - mx);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    with open(oracle.SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mpath = tmp_path / "mutant.cpp"
    mpath.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    subprocess.run(oracle.compile_command(str(mpath), lib_path), check=True)
    lib = oracle.load(lib_path)
    failed = []
    for check in CHECKS:
        try:
            check(lib)
        except (AssertionError, RuntimeError, ValueError):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
