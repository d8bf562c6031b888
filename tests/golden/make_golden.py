"""Writes the stored expected values under tests/golden/ that come from a
program. It calls only the CPU oracle (and the seeded input generator for the
inputs, which are stored beside the expected values).

config1_tiny.json: TP=2 virtual ranks, V=128 (shard 64 bf16 columns), cap=4,
M=1, three consecutive calls (parity 0, 1, 0). Call i uses input set i:
bf16(N(0,1)) from seed 0; each 32-bit word independently becomes the sentinel
pair (+0, -0) with probability 0.02, (+0, +0) with 0.01 and (-0, -0) with 0.01.

Run from the repository root:  python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from tp_vocab_logits_gb300 import synth  # noqa: E402


def words_hex(bits_u16: np.ndarray) -> list:
    w = np.ascontiguousarray(bits_u16).view(np.uint32)
    return [[f"0x{int(x):08X}" for x in row] for row in w.reshape(-1, w.shape[-1])]


def config1() -> dict:
    tp, W, cap, M = 2, 64, 4, 1
    g = oracle.Gather(tp, W, cap)
    calls = []
    for i in range(3):
        s = synth.shards(0, tp, M, W, sent_frac=0.02, zero_frac=0.01, negzero_frac=0.01,
                         set_index=i).numpy().view(np.uint16)
        before = g.parity
        out = g.call(s)
        calls.append({
            "M": M,
            "parity_before": before,
            "shards": [words_hex(s[r]) for r in range(tp)],
            "out": [words_hex(out[d]) for d in range(tp)],
            "parity_after": g.parity,
        })
    return {
        "about": __doc__.strip().split("\n\n")[1],
        "written_by": "tests/golden/make_golden.py (CPU oracle only)",
        "tp": tp, "shard_cols": W, "cap": cap,
        "calls": calls,
    }


if __name__ == "__main__":
    oracle.build()
    with open(os.path.join(HERE, "config1_tiny.json"), "w") as f:
        json.dump(config1(), f, indent=1)
    print("wrote config1_tiny.json")
