"""Runs the CPU oracle's quantizer on many matrices in parallel (test
infrastructure).  The pool is started with the `spawn` method, so its
workers are fresh interpreters that never touch the GPU (a process forked
after CUDA is initialised can hang)."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from oracle import int4g_oracle as O


def _quantize(W):
    return O.quantize(W)


def quantize_many(make, count, workers=None):
    """[canonical triple of make(i) for i < count]: the oracle's quantizer on
    each fp32 numpy matrix make(i) returns, in a spawn pool of `workers`
    processes (default: up to 12).  The matrices are made a few at a time,
    so that host memory holds only about two per worker."""
    if count == 0:
        return []
    n = workers or max(1, min(12, (os.cpu_count() or 2) - 1, count))
    if n == 1:
        return [_quantize(make(i)) for i in range(count)]
    out = []
    with mp.get_context("spawn").Pool(n) as pool:
        for c0 in range(0, count, 2 * n):
            mats = [make(i) for i in range(c0, min(count, c0 + 2 * n))]
            out += pool.map(_quantize, mats, chunksize=1)
            del mats
    return out
