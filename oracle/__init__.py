"""CPU oracle of the vocab-parallel logits gather (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg and reference arm of ``bench.py`` may use this package; the library under
``tp_vocab_logits_gb300`` never imports it and shares no code with it.

The arithmetic lives in ``hg_oracle.cpp`` (plain C++, compiled with g++); this
module only compiles it on demand and moves numpy arrays in and out.
Definition followed: the vLLM API page
"vllm.models.kimi_k3.nvidia.specialized_decode.runtime.logits_gather"
(class HeadGather) and the vLLM pull request "[Perf][Kimi-K3] Use the one-shot
custom all-gather for TP logits" (section "Purpose").
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "hg_oracle.cpp")
LIB = os.path.join(_HERE, "liboracle.so")


def compile_command(src: str = SRC, out: str = LIB, extra: tuple = ()) -> list:
    """g++ command line that builds the oracle shared library."""
    return ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", *extra, src, "-o", out]


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".{os.getpid()}.tmp"
        subprocess.run(compile_command(out=tmp), check=True)
        os.replace(tmp, LIB)
    return LIB


_u32p = ctypes.POINTER(ctypes.c_uint32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load an oracle library (the default one, built on demand)."""
    lib = ctypes.CDLL(path or build())
    lib.og_sentinel.restype = ctypes.c_uint32
    lib.og_create.restype = ctypes.c_void_p
    lib.og_create.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int]
    lib.og_destroy.argtypes = [ctypes.c_void_p]
    lib.og_parity.restype = ctypes.c_int
    lib.og_parity.argtypes = [ctypes.c_void_p]
    lib.og_mailbox.restype = _u32p
    lib.og_mailbox.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    lib.og_call.restype = ctypes.c_int
    lib.og_call.argtypes = [ctypes.c_void_p, ctypes.c_int, _u32p, _u32p]
    lib.og_slice_bf16.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p]
    lib.og_lm_head_f64.argtypes = [_u16p, _u16p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, _f64p]
    lib.og_row_stats.argtypes = [_u16p, ctypes.c_int, _f64p, _i32p, _f64p]
    return lib


_DEFAULT: ctypes.CDLL | None = None


def _lib() -> ctypes.CDLL:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = load()
    return _DEFAULT


def sentinel(lib: ctypes.CDLL | None = None) -> int:
    return int((lib or _lib()).og_sentinel())


class Gather:
    """Stateful oracle of one HeadGather: mailboxes of every virtual rank plus
    the parity. ``call`` takes the [tp, M, W] bf16 shards as uint16 bits and
    returns the [tp, M, V] outputs as uint16 bits."""

    def __init__(self, tp: int, shard_cols: int, cap: int, rows=None, lib=None):
        self._lib = lib or _lib()
        rows = list(rows or [])
        arr = (ctypes.c_int * max(1, len(rows)))(*rows)
        self._h = self._lib.og_create(tp, shard_cols, cap, arr, len(rows))
        if not self._h:
            raise ValueError(f"oracle rejects tp={tp} shard_cols={shard_cols} cap={cap} rows={rows}")
        self.tp, self.W, self.cap = tp, shard_cols, cap
        self.V = tp * shard_cols

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.og_destroy(h)
            self._h = None

    @property
    def parity(self) -> int:
        return int(self._lib.og_parity(self._h))

    def mailbox(self, d: int, q: int) -> np.ndarray:
        """Copy of rank d's mailbox, parity q: [cap, V/2] uint32 words."""
        p = self._lib.og_mailbox(self._h, d, q)
        n = self.cap * self.V // 2
        return np.ctypeslib.as_array(p, shape=(n,)).copy().reshape(self.cap, self.V // 2)

    def call_status(self, shards_bits: np.ndarray):
        """(status, out) for one call; out is None unless status == 0."""
        s = np.ascontiguousarray(shards_bits, dtype=np.uint16)
        tp, M, W = s.shape
        assert tp == self.tp and W == self.W
        words = s.view(np.uint32)
        out = np.empty((tp, M, self.V // 2), dtype=np.uint32)
        st = self._lib.og_call(self._h, M, words.ctypes.data_as(_u32p), out.ctypes.data_as(_u32p))
        return int(st), (out.view(np.uint16).reshape(tp, M, self.V) if st == 0 else None)

    def call(self, shards_bits: np.ndarray) -> np.ndarray:
        st, out = self.call_status(shards_bits)
        if st != 0:
            raise RuntimeError(f"oracle call failed with status {st}")
        return out


def slice_vocab(out_bits: np.ndarray, v_real: int, lib=None) -> np.ndarray:
    """Padded-vocab slice of one [M, V] bf16 output (uint16 bits)."""
    o = np.ascontiguousarray(out_bits, dtype=np.uint16)
    M, V = o.shape
    res = np.empty((M, v_real), dtype=np.uint16)
    (lib or _lib()).og_slice_bf16(o.ctypes.data_as(_u16p), M, V, v_real, res.ctypes.data_as(_u16p))
    return res


def lm_head_f64(hidden_bits: np.ndarray, weight_bits: np.ndarray, n0: int = 0,
                n1: int | None = None, lib=None) -> np.ndarray:
    """Double-precision logits of one rank for vocab columns [n0, n1):
    hidden [M, K] and weight [W, K] as bf16 bits; returns [M, n1 - n0] float64."""
    h = np.ascontiguousarray(hidden_bits, dtype=np.uint16)
    wt = np.ascontiguousarray(weight_bits, dtype=np.uint16)
    M, K = h.shape
    W, K2 = wt.shape
    assert K == K2
    n1 = W if n1 is None else n1
    assert 0 <= n0 <= n1 <= W
    res = np.empty((M, n1 - n0), dtype=np.float64)
    (lib or _lib()).og_lm_head_f64(h.ctypes.data_as(_u16p), wt.ctypes.data_as(_u16p), M, K,
                                   n0, n1, res.ctypes.data_as(_f64p))
    return res


def row_stats(row_bits: np.ndarray, lib=None) -> tuple:
    """(max_logit, argmax, sum_exp) of one gathered bf16 row (uint16 bits)."""
    r = np.ascontiguousarray(row_bits, dtype=np.uint16)
    mx, s = ctypes.c_double(), ctypes.c_double()
    arg = ctypes.c_int()
    (lib or _lib()).og_row_stats(r.ctypes.data_as(_u16p), r.shape[0], ctypes.byref(mx),
                                 ctypes.byref(arg), ctypes.byref(s))
    return mx.value, arg.value, s.value
