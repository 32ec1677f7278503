"""CPU oracle for GGUF block-quantized mul_mat — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
leg may import this package.  The library path never does.  It shares no code with the
CUDA path: the arithmetic lives in ``syn_oracle.c`` (plain scalar C, ``-ffp-contract=off``)
and this module only marshals numpy arrays into it.

Sources: "The GGML ecosystem, and where synapse fits", section 5 (the block-format table
and "Products: weights against quantized activations"); yakaai ggml documentation,
examples/simple (ggml_mul_mat(A, B^T) = C^T).

Parity status per function (see the tests under tests/test_oracle_*.py for the pins):
  fp16 conversion        pinned (numpy.float16 on a dense sample, boundaries exhaustive)
  quantize Q8_0/Q8_K     pinned (hand blocks, error bound, fixed point, bsum invariant)
  quantize Q4_K/Q6_K     pinned to hand-worked super-blocks (tests/golden/q4_k_worked.txt,
                         q6_k_worked.txt: super-scales, every sub-block scale and min, every
                         code, with rounding ties and clamps) and to the closed-form error
                         bounds; the encoders are the plain readings of the format table
  quantize Q4_0/Q5_0     pinned to error bounds, the exact extreme, hand blocks
  F16 weights            pinned (the fp16 conversion; the product against numpy float16 casts)
  dequantize             pinned (hand-written block bytes against the format formulas)
  block sums / mul_mat   pinned (fp64 brute force over dequantized blocks, the
                         ggml_mul_mat orientation example with exact integers)
  byte layout in blocks  unpinnable here (no GGUF file or gguf-py); it is the public
                         GGUF layout, written down in syn_oracle.c
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q8_0, Q4_K, Q6_K, Q8_K, Q4_0, Q5_0, F16 = 1, 2, 3, 4, 5, 6, 7
BLOCK_ELEMS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, Q8_K: 256, Q4_0: 32, Q5_0: 32, F16: 1}
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, Q8_K: 292, Q4_0: 18, Q5_0: 22, F16: 2}
VEC_DOT_TYPE = {Q8_0: Q8_0, Q4_K: Q8_K, Q6_K: Q8_K, Q4_0: Q8_0, Q5_0: Q8_0, F16: F16}
NAMES = {Q8_0: "Q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K", Q8_K: "Q8_K", Q4_0: "Q4_0", Q5_0: "Q5_0", F16: "F16"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "syn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile syn_oracle.c into oracle/_build/liboracle.so (gcc, -O2, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            L.orc_fp32_to_fp16.argtypes = [ctypes.c_float]
            L.orc_fp32_to_fp16.restype = ctypes.c_uint16
            L.orc_fp16_to_fp32.argtypes = [ctypes.c_uint16]
            L.orc_fp16_to_fp32.restype = ctypes.c_float
            L.orc_fp32_to_fp16_array.argtypes = [vp, vp, i64]
            L.orc_fp16_to_fp32_array.argtypes = [vp, vp, i64]
            L.orc_block_elems.argtypes = [i32]
            L.orc_block_elems.restype = i64
            L.orc_block_bytes.argtypes = [i32]
            L.orc_block_bytes.restype = i64
            L.orc_vec_dot_type.argtypes = [i32]
            L.orc_vec_dot_type.restype = i32
            L.orc_quantize.argtypes = [i32, vp, vp, i64, i64]
            L.orc_quantize.restype = i32
            L.orc_dequantize.argtypes = [i32, vp, vp, i64, i64]
            L.orc_dequantize.restype = i32
            L.orc_unpack_q4_k.argtypes = [vp, vp, vp, vp, vp, vp]
            L.orc_unpack_q6_k.argtypes = [vp, vp, vp, vp]
            L.orc_unpack_qx_0.argtypes = [i32, vp, vp, vp]
            L.orc_unpack_qx_0.restype = i32
            L.orc_block_sums.argtypes = [i32, vp, i64, i64, vp, i64, vp]
            L.orc_block_sums.restype = i32
            L.orc_mul_mat.argtypes = [i32, vp, i64, i64, vp, i64, vp, i32]
            L.orc_mul_mat.restype = i32
            L.orc_mul_mat_sampled.argtypes = [i32, vp, i64, i64, vp, i64, vp, i64, vp, i64, vp]
            L.orc_mul_mat_sampled.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(st: int, what: str):
    if st != 0:
        raise OracleError(f"{what}: oracle status {st}")


def row_bytes(t: int, n: int) -> int:
    return (n // BLOCK_ELEMS[t]) * BLOCK_BYTES[t]


def fp32_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_fp32_to_fp16_array(_p(x), _p(out), x.size)
    return out


def fp16_bits_to_fp32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().orc_fp16_to_fp32_array(_p(h), _p(out), h.size)
    return out


def quantize(t: int, x: np.ndarray) -> np.ndarray:
    """fp32 (n_rows, n_per_row) -> uint8 (n_rows, row_bytes).  Raises on range errors."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    n_rows, n = x.shape
    out = np.zeros((n_rows, row_bytes(t, n)), dtype=np.uint8)
    _check(lib().orc_quantize(t, _p(x), _p(out), n_rows, n), "quantize")
    return out


def quantize_status(t: int, x: np.ndarray) -> int:
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    n_rows, n = x.shape
    out = np.zeros((n_rows, max(row_bytes(t, n), 1)), dtype=np.uint8)
    return lib().orc_quantize(t, _p(x), _p(out), n_rows, n)


def dequantize(t: int, q: np.ndarray, n_per_row: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    n_rows = q.size // row_bytes(t, n_per_row)
    out = np.empty((n_rows, n_per_row), dtype=np.float32)
    _check(lib().orc_dequantize(t, _p(q), _p(out), n_rows, n_per_row), "dequantize")
    return out


def unpack_q4_k(block: np.ndarray):
    block = np.ascontiguousarray(block, dtype=np.uint8)
    d = np.zeros(1, np.uint16); dm = np.zeros(1, np.uint16)
    sc = np.zeros(8, np.uint8); mn = np.zeros(8, np.uint8); q = np.zeros(256, np.uint8)
    lib().orc_unpack_q4_k(_p(block), _p(d), _p(dm), _p(sc), _p(mn), _p(q))
    return int(d[0]), int(dm[0]), sc, mn, q


def unpack_q6_k(block: np.ndarray):
    block = np.ascontiguousarray(block, dtype=np.uint8)
    d = np.zeros(1, np.uint16); sc = np.zeros(16, np.int8); q = np.zeros(256, np.uint8)
    lib().orc_unpack_q6_k(_p(block), _p(d), _p(sc), _p(q))
    return int(d[0]), sc, q


def unpack_qx_0(t: int, block: np.ndarray):
    """Q4_0 / Q5_0 block -> (d bits, 32 codes)."""
    block = np.ascontiguousarray(block, dtype=np.uint8)
    d = np.zeros(1, np.uint16); q = np.zeros(32, np.uint8)
    _check(lib().orc_unpack_qx_0(t, _p(block), _p(d), _p(q)), "unpack_qx_0")
    return int(d[0]), q


def quantize_activations(wtype: int, x: np.ndarray) -> np.ndarray:
    """Activation rows in the vec_dot_type of weight format wtype (packed blocks)."""
    return quantize(VEC_DOT_TYPE[wtype], x)


def block_sums(wtype: int, W: np.ndarray, n_out: int, n_in: int, Xq: np.ndarray, n_tok: int) -> np.ndarray:
    """int32 (n_tok, n_out, n_blocks, 2): Q8_0 [I, 0]; Q4_K [A, Bm]; Q6_K [C, 0]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    nb = n_in // BLOCK_ELEMS[wtype]
    S = np.zeros((n_tok, n_out, nb, 2), dtype=np.int32)
    _check(lib().orc_block_sums(wtype, _p(W), n_out, n_in, _p(Xq), n_tok, _p(S)), "block_sums")
    return S


def mul_mat(wtype: int, W: np.ndarray, n_out: int, n_in: int, X: np.ndarray, n_threads: int = 1) -> np.ndarray:
    """Y (n_tok, n_out) fp32 = ggml_mul_mat(W, X): X quantized to the vec_dot_type first."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    X = np.ascontiguousarray(X, dtype=np.float32)
    if X.ndim == 1:
        X = X[None, :]
    n_tok = X.shape[0]
    Y = np.zeros((n_tok, n_out), dtype=np.float32)
    _check(lib().orc_mul_mat(wtype, _p(W), n_out, n_in, _p(X), n_tok, _p(Y), n_threads), "mul_mat")
    return Y


def mul_mat_sampled(wtype: int, W: np.ndarray, n_out: int, n_in: int, X: np.ndarray,
                    rows: np.ndarray, toks: np.ndarray) -> np.ndarray:
    """Y[toks][:, rows] of mul_mat, computed only at the sampled entries."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    X = np.ascontiguousarray(X, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    toks = np.ascontiguousarray(toks, dtype=np.int64)
    Ys = np.zeros((toks.size, rows.size), dtype=np.float32)
    _check(lib().orc_mul_mat_sampled(wtype, _p(W), n_out, n_in, _p(X), X.shape[0],
                                     _p(rows), rows.size, _p(toks), toks.size, _p(Ys)),
           "mul_mat_sampled")
    return Ys
