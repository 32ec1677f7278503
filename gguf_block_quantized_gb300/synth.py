"""Seeded synthetic inputs, shared by the tests, the smoke check and the benchmark.

Holds random-number generation only — none of the method's arithmetic.  Weights are
~N(0, 0.02) and activations ~N(0, 1), drawn as fp32 with numpy's PCG64 ``default_rng``.
Seeds follow ``1000*workload + 2*tensor_index`` for a weight and ``+1`` for its
activations, so that every consumer sees the same host arrays.
"""
from __future__ import annotations

import numpy as np

W_STD = 0.02
X_STD = 1.0


def normal(seed: int, shape, std: float = 1.0) -> np.ndarray:
    a = np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def weight(workload: int, index: int, n_out: int, n_in: int) -> np.ndarray:
    return normal(1000 * workload + 2 * index, (n_out, n_in), W_STD)


def activations(workload: int, index: int, n_tok: int, n_in: int) -> np.ndarray:
    return normal(1000 * workload + 2 * index + 1, (n_tok, n_in), X_STD)


def uniform(seed: int, shape, lo: float, hi: float) -> np.ndarray:
    return np.random.default_rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def integers(seed: int, shape, lo: int, hi: int, dtype=np.int64) -> np.ndarray:
    return np.random.default_rng(seed).integers(lo, hi, size=shape, dtype=dtype)
