"""Seeded synthetic inputs, shared by the tests, the smoke check and the benchmark.

Holds random-number generation only — none of the method's arithmetic.  Weights are
~N(0, 0.02) and activations ~N(0, 1), drawn as fp32 with numpy's PCG64 ``default_rng``.
Seeds follow ``1000*workload + 2*tensor_index`` for a weight and ``+1`` for its
activations, so that every consumer sees the same host arrays.  A weight matrix is drawn
in chunks of WEIGHT_CHUNK_ROWS rows, chunk c from ``default_rng((seed, c))``: any rows
can be drawn on their own, and the chunks of a large matrix in parallel threads (the
generator releases the GIL while it fills an array), which keeps the 4.1e9 weights of the
Llama-8B sweep to seconds of host time.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

WEIGHT_CHUNK_ROWS = 256

W_STD = 0.02
X_STD = 1.0


def normal(seed: int, shape, std: float = 1.0) -> np.ndarray:
    a = np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def weight_rows(workload: int, index: int, n_in: int, chunk: int, n_out: int, n_rows: int | None = None) -> np.ndarray:
    """Rows [chunk*WEIGHT_CHUNK_ROWS, ...) of weight(workload, index, n_out, n_in); with n_rows,
    only the first n_rows of them (the generator fills rows in order)."""
    r0 = chunk * WEIGHT_CHUNK_ROWS
    n = min(WEIGHT_CHUNK_ROWS, n_out - r0) if n_rows is None else min(n_rows, WEIGHT_CHUNK_ROWS, n_out - r0)
    a = np.random.default_rng((1000 * workload + 2 * index, chunk)).standard_normal(
        size=(n, n_in), dtype=np.float32)
    a *= np.float32(W_STD)
    return a


def weight(workload: int, index: int, n_out: int, n_in: int) -> np.ndarray:
    out = np.empty((n_out, n_in), np.float32)
    n_chunks = -(-n_out // WEIGHT_CHUNK_ROWS)

    def fill(c):
        r0 = c * WEIGHT_CHUNK_ROWS
        out[r0:r0 + WEIGHT_CHUNK_ROWS] = weight_rows(workload, index, n_in, c, n_out)

    if n_out * n_in < (1 << 22):
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


def activations(workload: int, index: int, n_tok: int, n_in: int) -> np.ndarray:
    return normal(1000 * workload + 2 * index + 1, (n_tok, n_in), X_STD)


def uniform(seed: int, shape, lo: float, hi: float) -> np.ndarray:
    return np.random.default_rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def integers(seed: int, shape, lo: int, hi: int, dtype=np.int64) -> np.ndarray:
    return np.random.default_rng(seed).integers(lo, hi, size=shape, dtype=dtype)
