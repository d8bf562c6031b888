"""Shared helpers of the GPU tests: moving bf16 bit patterns between numpy
(oracle side) and torch device tensors (library side)."""

import numpy as np
import torch

S_I32 = -(1 << 31)  # 0x80000000 as int32


def to_dev(bits_u16: np.ndarray) -> list:
    """[tp, M, W] uint16 -> list of tp contiguous int16 device tensors."""
    t = torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).cuda()
    return [t[r].contiguous() for r in range(t.shape[0])]


def from_dev(ts) -> np.ndarray:
    """list of [M, V] int16 device tensors -> [tp, M, V] uint16 numpy."""
    return torch.stack(list(ts)).cpu().numpy().view(np.uint16)


def empty_outs(tp: int, M: int, V: int, fill: int = 0x5A5A) -> list:
    return [torch.full((M, V), fill - (1 << 16) if fill >= (1 << 15) else fill,
                       dtype=torch.int16, device="cuda") for _ in range(tp)]


def assert_mailboxes_armed(h, hg) -> None:
    for d in range(h.tp):
        mb = hg.mailbox_words(h, d)
        bad = (mb != S_I32).sum().item()
        assert bad == 0, f"rank {d}: {bad} mailbox words are not the sentinel"


def rewrite_concat(shards) -> torch.Tensor:
    """The gather's expected row block written with torch ops: rank-order
    concat of the shards' 32-bit words, the sentinel word sent as zero."""
    words = torch.cat([s.view(torch.int32) for s in shards], dim=1)
    return torch.where(words == S_I32, torch.zeros_like(words), words)
