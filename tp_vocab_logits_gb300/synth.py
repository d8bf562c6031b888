"""Seeded synthetic inputs for the logits gather and the LM-head producer.

This module only makes inputs. It holds none of the gather's or the LM head's
arithmetic, and it is the one piece of code that both the CUDA path's tests
and the CPU oracle's tests use, so that both sides see identical bytes.

Generator: counter-based splitmix64 (S. Vigna's published finaliser; the
stream key is the finaliser applied to the seed and a stream id). Element
(set, rank, row, col) of a tensor kind uses the counter built from those
indices at fixed bit offsets, so a value depends only on its indices and never
on the tensor's shape: any slice can be regenerated alone, on the CPU or on
the GPU, and comes out the same. Normal samples use Box-Muller on two
independent uniform streams; values are rounded to bf16 by torch's
float32 -> bfloat16 conversion (round to nearest even).

The implementation uses torch int64 arithmetic only (wrapping multiplication,
masked right shifts), so the same code runs on any device.
"""

from __future__ import annotations

import math

import torch

# splitmix64 constants, as signed int64 two's-complement values.
_GAMMA = 0x9E3779B97F4A7C15 - (1 << 64)
_MUL1 = 0xBF58476D1CE4E5B9 - (1 << 64)
_MUL2 = 0x94D049BB133111EB - (1 << 64)

# Word of the BF16 pair (+0, -0): +0 (0x0000) in the low half, -0 (0x8000) in
# the high half. Inputs inject it to exercise the gather's sentinel handling.
PAIR_POS_NEG_ZERO = 0x80000000
PAIR_POS_POS_ZERO = 0x00000000
PAIR_NEG_NEG_ZERO = 0x80008000
BF16_NEG_INF = 0xFF80

# Further 32-bit words next to the sentinel, injected on request (extra_frac):
# the pair (-0, +0) (the sentinel's halves swapped), words one bit away from
# the sentinel (lowest bit; lowest bit of the high half; the bit below the
# sign), a NaN pair, and the pairs (-inf, -inf) and (+inf, +inf). None of
# them is the sentinel, so each must move unchanged.
EXTRA_WORDS = (0x00008000, 0x80000001, 0x80010000, 0xC0000000, 0x7FC07FC0, 0xFF80FF80,
               0x7F807F80)

# Stream ids (one per use of randomness).
_S_U1, _S_U2, _S_INJECT, _S_EXTRA, _S_EXTRA_PICK = 1, 2, 3, 4, 5
# Tensor kinds, folded into the key so that kinds never share a stream.
KIND_SHARD, KIND_HIDDEN, KIND_WEIGHT, KIND_SEQUENCE = 1, 2, 3, 4


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _MUL1
    z = (z ^ _srl(z, 27)) * _MUL2
    return z ^ _srl(z, 31)


def _mix_int(z: int) -> int:
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def _key(seed: int, kind: int, stream: int) -> int:
    k = _mix_int(_mix_int(seed * 0x9E3779B97F4A7C15 + 0x632BE59BD9B4E019) + (kind << 8) + stream)
    return k - (1 << 64) if k >= (1 << 63) else k


def _uniform(counter: torch.Tensor, seed: int, kind: int, stream: int) -> torch.Tensor:
    """float64 uniforms in [0, 1) with 53 random bits."""
    z = _mix((counter + 1) * _GAMMA + _key(seed, kind, stream))
    return _srl(z, 11).to(torch.float64) * (2.0 ** -53)


def _normal(counter: torch.Tensor, seed: int, kind: int) -> torch.Tensor:
    u1 = _uniform(counter, seed, kind, _S_U1)
    u2 = _uniform(counter, seed, kind, _S_U2)
    r = torch.sqrt(-2.0 * torch.log1p(-u1))  # 1 - u1 is in (0, 1]
    return r * torch.cos((2.0 * math.pi) * u2)


def _to_bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """bf16 bit patterns (int16) of float64 values via float32."""
    return x.to(torch.float32).to(torch.bfloat16).view(torch.int16)


def _grid(shape, shifts, offsets, device) -> torch.Tensor:
    """counter[i0, i1, ...] = sum_k (offset_k + i_k) << shift_k."""
    c = torch.zeros((), dtype=torch.int64, device=device)
    nd = len(shape)
    for k, (n, s, o) in enumerate(zip(shape, shifts, offsets)):
        idx = (torch.arange(n, dtype=torch.int64, device=device) + o) << s
        c = c + idx.view([n if i == k else 1 for i in range(nd)])
    return c


def shards(seed: int, tp: int, M: int, W: int, *, dist: str = "normal", scale: float = 1.0,
           sent_frac: float = 0.0, zero_frac: float = 0.0, negzero_frac: float = 0.0,
           extra_frac: float = 0.0, set_index: int = 0, rank0: int = 0, row0: int = 0,
           col0: int = 0, v_real: int | None = None, device="cpu") -> torch.Tensor:
    """Logits shards of tp virtual ranks as bf16 bits: int16 [tp, M, W].

    dist "normal": bf16(N(0, scale^2)); dist "uniform": bf16(U(-scale, scale)).
    Then each 32-bit word (bf16 columns 2k, 2k+1) independently becomes, with
    probability sent_frac, the pair (+0, -0); with probability zero_frac the
    pair (+0, +0); with probability negzero_frac the pair (-0, -0). After
    that, each word independently becomes, with probability extra_frac, one of
    EXTRA_WORDS, each of them equally likely (separate random streams: with
    extra_frac 0 the result is the same as without it).
    v_real: real vocab width of a padded vocab; columns at or beyond it of the
    full [M, tp*W] row hold bf16 -inf.
    rank0/row0/col0 offset the indices, so a slice of a larger tensor can be
    generated alone. Indices: set < 2^11, rank < 2^8, row < 2^12, col < 2^20.
    """
    assert W % 2 == 0 and col0 % 2 == 0
    assert set_index < (1 << 11) and rank0 + tp <= (1 << 8)
    assert row0 + M <= (1 << 12) and col0 + W <= (1 << 20)
    base = set_index << 52
    cnt = _grid((tp, M, W), (44, 32, 0), (rank0, row0, col0), device) + base
    if dist == "normal":
        vals = _normal(cnt, seed, KIND_SHARD) * scale
    elif dist == "uniform":
        vals = (_uniform(cnt, seed, KIND_SHARD, _S_U1) * 2.0 - 1.0) * scale
    else:
        raise ValueError(dist)
    bits = _to_bf16_bits(vals)
    words = bits.view(torch.int32)  # [tp, M, W/2] little-endian pairs
    if sent_frac or zero_frac or negzero_frac:
        wcnt = _grid((tp, M, W // 2), (44, 32, 0), (rank0, row0, col0 // 2), device) + base
        u = _uniform(wcnt, seed, KIND_SHARD, _S_INJECT)
        t1 = sent_frac
        t2 = t1 + zero_frac
        t3 = t2 + negzero_frac
        def as_i32(v):
            return torch.tensor(v - (1 << 32) if v >= (1 << 31) else v, dtype=torch.int32,
                                device=device)
        words = torch.where(u < t1, as_i32(PAIR_POS_NEG_ZERO), words)
        words = torch.where((u >= t1) & (u < t2), as_i32(PAIR_POS_POS_ZERO), words)
        words = torch.where((u >= t2) & (u < t3), as_i32(PAIR_NEG_NEG_ZERO), words)
        bits = words.view(torch.int16).view(tp, M, W)
    if extra_frac:
        words = bits.view(torch.int32)
        wcnt = _grid((tp, M, W // 2), (44, 32, 0), (rank0, row0, col0 // 2), device) + base
        u = _uniform(wcnt, seed, KIND_SHARD, _S_EXTRA)
        pick = (_uniform(wcnt, seed, KIND_SHARD, _S_EXTRA_PICK) * len(EXTRA_WORDS)).to(torch.int64)
        pick = torch.clamp(pick, max=len(EXTRA_WORDS) - 1)
        table = torch.tensor([v - (1 << 32) if v >= (1 << 31) else v for v in EXTRA_WORDS],
                             dtype=torch.int32, device=device)
        words = torch.where(u < extra_frac, table[pick], words)
        bits = words.view(torch.int16).view(tp, M, W)
    if v_real is not None:
        col = (torch.arange(tp, device=device).view(tp, 1, 1) + rank0) * W \
            + torch.arange(W, device=device).view(1, 1, W) + col0
        bits = torch.where(col >= v_real, torch.tensor(BF16_NEG_INF - (1 << 16), dtype=torch.int16,
                                                        device=device), bits)
    return bits.contiguous()


def hidden(seed: int, tp: int, M: int, K: int, *, device="cpu") -> torch.Tensor:
    """LM-head inputs of tp virtual ranks: bf16(N(0, 1)) bits, int16 [tp, M, K]."""
    assert tp <= (1 << 8) and M <= (1 << 12) and K <= (1 << 20)
    cnt = _grid((tp, M, K), (44, 32, 0), (0, 0, 0), device)
    return _to_bf16_bits(_normal(cnt, seed, KIND_HIDDEN)).contiguous()


def weight(seed: int, rank: int, W: int, K: int, *, std: float = 0.02, row0: int = 0,
           device="cpu") -> torch.Tensor:
    """LM-head weight of one virtual rank in the nn.Linear layout [W, K]
    (vocab rows, hidden columns): bf16(N(0, std^2)) bits, int16 [W, K].
    row0 offsets the vocab index, so any block of rows can be generated alone."""
    assert rank < (1 << 8) and row0 + W <= (1 << 24) and K <= (1 << 20)
    cnt = _grid((W, K), (20, 0), (row0, 0), device) + (rank << 44)
    return _to_bf16_bits(_normal(cnt, seed, KIND_WEIGHT) * std).contiguous()


def row_sequence(seed: int, n: int, choices) -> list:
    """A seeded sequence of n row counts drawn uniformly from choices."""
    cnt = torch.arange(n, dtype=torch.int64)
    u = _uniform(cnt, seed, KIND_SEQUENCE, _S_U1)
    idx = torch.clamp((u * len(choices)).to(torch.int64), max=len(choices) - 1)
    return [int(choices[i]) for i in idx.tolist()]
