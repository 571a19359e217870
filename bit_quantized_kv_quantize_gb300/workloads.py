"""Seeded synthetic workloads shaped like the pages' Llama-2 / Llama-3 caches.

This module draws inputs only; it holds none of the method's arithmetic, so
both the CUDA path (tests, benchmark) and the CPU oracle take their inputs
from here.  Every tensor is a pure function of (config, seed, stream), drawn
with numpy's counter-based Philox generator, so any (sequence, head) slice
can be regenerated on its own without drawing the rest.

Values are N(0, 1) in fp32, rounded to fp16 (round-half-to-even by numpy).
Keys get per-(sequence, kv head) outlier channels scaled by a factor before
the fp16 rounding (the channel-outlier structure that motivates per-channel
key quantization in the KIVI section, core algorithm item 2).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    b: int
    h_q: int
    h_kv: int
    d: int
    kbits: int
    vbits: int
    G: int
    R: int
    prefill: int            # prefill tokens per sequence (max when ragged)
    steps: int              # decode steps (append + attention)
    n_outlier: int          # outlier key channels per kv head
    outlier_scale: float
    ragged: tuple = ()      # (low, high) inclusive: prefill lengths drawn uniformly
    seed: int = 0

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    def capacity(self) -> int:
        return self.prefill + self.steps

    def lengths(self) -> np.ndarray:
        """Prefill length of every sequence."""
        if not self.ragged:
            return np.full(self.b, self.prefill, np.int32)
        rng = np.random.default_rng(self.seed)
        lo, hi = self.ragged
        return rng.integers(lo, hi + 1, size=self.b).astype(np.int32)


def _outliers(d):
    return int(round(0.02 * d))


# The five workloads: tiny reference case, Llama-2-7B layer, Llama-3-8B GQA at
# 32k, KIVI-4 ragged serving batch, 128k long context.
WORKLOADS = {
    "tiny_kivi2": Workload("tiny_kivi2", b=1, h_q=2, h_kv=2, d=64, kbits=2, vbits=2, G=32, R=32,
                           prefill=256, steps=64, n_outlier=4, outlier_scale=10.0),
    "llama2_7b_4k": Workload("llama2_7b_4k", b=1, h_q=32, h_kv=32, d=128, kbits=2, vbits=2, G=32,
                             R=128, prefill=4096, steps=1, n_outlier=_outliers(128),
                             outlier_scale=8.0),
    "llama3_8b_gqa_32k": Workload("llama3_8b_gqa_32k", b=8, h_q=32, h_kv=8, d=128, kbits=2,
                                  vbits=2, G=32, R=128, prefill=32767, steps=1,
                                  n_outlier=_outliers(128), outlier_scale=8.0),
    "kivi4_serving": Workload("kivi4_serving", b=64, h_q=32, h_kv=8, d=128, kbits=4, vbits=4,
                              G=32, R=128, prefill=4096, steps=256, n_outlier=0,
                              outlier_scale=1.0, ragged=(1024, 4096)),
    "long_128k": Workload("long_128k", b=1, h_q=32, h_kv=8, d=128, kbits=2, vbits=2, G=32, R=128,
                          prefill=131071, steps=1, n_outlier=_outliers(128), outlier_scale=10.0),
}

_KIND = {"K": 1, "V": 2, "q": 3, "k_new": 4, "v_new": 5, "outlier": 6, "Q": 7}


def _gen(seed: int, kind: str, a: int, b: int = 0) -> np.random.Generator:
    key = np.array([np.uint64(seed), np.uint64((_KIND[kind] << 56) | (a << 28) | b)], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def outlier_channels(w: Workload, seq: int, head: int) -> np.ndarray:
    if w.n_outlier == 0:
        return np.zeros(0, np.int64)
    return np.sort(_gen(w.seed, "outlier", seq, head).choice(w.d, w.n_outlier, replace=False))


def _keys_fp16(w: Workload, x: np.ndarray, seq: int, head: int) -> np.ndarray:
    ch = outlier_channels(w, seq, head)
    if ch.size:
        x[..., ch] *= np.float32(w.outlier_scale)
    return x.astype(np.float16)


def prefill_slice(w: Workload, kind: str, seq: int, head: int, n: int) -> np.ndarray:
    """First n prefill tokens of one (sequence, kv head): fp16 [n, d]."""
    x = _gen(w.seed, kind, seq, head).standard_normal((n, w.d), dtype=np.float32)
    return _keys_fp16(w, x, seq, head) if kind == "K" else x.astype(np.float16)


def prefill_kv(w: Workload, t_stride: int | None = None, threads: int | None = None,
               seqs=None):
    """K, V fp16 [b, h_kv, t_stride, d] and the per-sequence lengths.

    Tokens past a sequence's length are zero.  With ``seqs``, only those
    sequences are drawn (the others stay zero)."""
    lens = w.lengths()
    t_stride = int(t_stride or lens.max() or 1)
    K = np.zeros((w.b, w.h_kv, t_stride, w.d), np.float16)
    V = np.zeros_like(K)
    todo = [(i, j) for i in (range(w.b) if seqs is None else seqs) for j in range(w.h_kv)]

    def fill(ij):
        i, j = ij
        n = int(lens[i])
        K[i, j, :n] = prefill_slice(w, "K", i, j, n)
        V[i, j, :n] = prefill_slice(w, "V", i, j, n)

    nthreads = threads or min(16, os.cpu_count() or 1)
    if nthreads > 1 and len(todo) > 1:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(fill, todo))
    else:
        for ij in todo:
            fill(ij)
    return K, V, lens


def prefill_q(w: Workload, t_stride: int | None = None, threads: int | None = None):
    """The prompt's queries: fp16 [b, h_q, t_stride, d], N(0, 1) per element,
    tokens past a sequence's length zero (inputs of the prefill attention)."""
    lens = w.lengths()
    t_stride = int(t_stride or lens.max() or 1)
    Q = np.zeros((w.b, w.h_q, t_stride, w.d), np.float16)

    def fill(ih):
        i, h = ih
        n = int(lens[i])
        Q[i, h, :n] = _gen(w.seed, "Q", i, h).standard_normal((n, w.d), dtype=np.float32).astype(np.float16)

    todo = [(i, h) for i in range(w.b) for h in range(w.h_q)]
    nthreads = threads or min(16, os.cpu_count() or 1)
    if nthreads > 1 and len(todo) > 1:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(fill, todo))
    else:
        for ih in todo:
            fill(ih)
    return Q


def step_kv(w: Workload, step: int):
    """New key and value of decode step ``step``: fp16 [b, h_kv, d] each."""
    k = _gen(w.seed, "k_new", step).standard_normal((w.b, w.h_kv, w.d), dtype=np.float32)
    for i in range(w.b):
        for j in range(w.h_kv):
            ch = outlier_channels(w, i, j)
            if ch.size:
                k[i, j, ch] *= np.float32(w.outlier_scale)
    v = _gen(w.seed, "v_new", step).standard_normal((w.b, w.h_kv, w.d), dtype=np.float32)
    return k.astype(np.float16), v.astype(np.float16)


def step_q(w: Workload, step: int) -> np.ndarray:
    """Query of decode step ``step``: fp16 [b, h_q, d]."""
    return _gen(w.seed, "q", step).standard_normal((w.b, w.h_q, w.d), dtype=np.float32).astype(np.float16)


def small(w: Workload, **kw) -> Workload:
    """The same workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **kw)
