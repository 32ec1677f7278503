"""Thin ctypes binding of libsyn.so (include/syn.h) — argument marshalling only.

Every function named ``syn_*`` mirrors the C entry point of the same name and takes raw
device pointers (ints) and a raw ``cudaStream_t`` (int, 0 = legacy default stream).
The helpers below them (``quantize``, ``dequantize``, ``quantize_activations``,
``mul_mat``, ``block_sums``) take torch CUDA tensors, allocate outputs with torch and
call the same entry points on torch's current stream.  There is no fallback: if the
library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsyn.so")

Q8_0, Q4_K, Q6_K, Q8_K, Q4_0, Q5_0, F16 = 1, 2, 3, 4, 5, 6, 7
OK, ERR_TYPE, ERR_SHAPE, ERR_NULL, ERR_ALIGN, ERR_RANGE, ERR_CUDA, ERR_TIMEOUT, ERR_NOMEM, ERR_DEVICE = \
    0, -1, -2, -3, -4, -5, -6, -7, -8, -9
ERR_TOO_LARGE = -10
STATIC_SCRATCH_BYTES = 32 << 20
BLOCK_ELEMS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, Q8_K: 256, Q4_0: 32, Q5_0: 32, F16: 1}
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, Q8_K: 292, Q4_0: 18, Q5_0: 22, F16: 2}
VEC_DOT_TYPE = {Q8_0: Q8_0, Q4_K: Q8_K, Q6_K: Q8_K, Q4_0: Q8_0, Q5_0: Q8_0, F16: F16}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libsyn.so is not built ({LIB_PATH}); run "
                      "`python -m gguf_block_quantized_gb300.build` (nvcc, sm_103a)")

_L = ctypes.CDLL(LIB_PATH)
_i64, _i32, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p

# (name, restype, argtypes): the declarations of include/syn.h
EXPORTS = [
    ("syn_block_elems", _i64, [_i32]),
    ("syn_block_bytes", _i64, [_i32]),
    ("syn_row_bytes", _i64, [_i32, _i64]),
    ("syn_quantize", _i32, [_i32, _vp, _vp, _i64, _i64, _vp]),
    ("syn_dequantize", _i32, [_i32, _vp, _vp, _i64, _i64, _vp]),
    ("syn_quantize_activations", _i32, [_i32, _vp, _i64, _i64, _vp, _vp, _vp, _vp]),
    ("syn_mul_mat", _i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    ("syn_reserve", _i32, [_i64, _i64, _vp]),
    ("syn_release", _i32, []),
    ("syn_block_sums", _i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    ("syn_set_gemv_max_tok", _i32, [_i32]),
    ("syn_device_status", _i32, [_i32]),
    ("syn_launch_count", _i64, []),
    ("syn_strerror", ctypes.c_char_p, [_i32]),
    ("syn_mul_mat_prefill_static", _i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
]

class MatDesc(ctypes.Structure):
    """syn_mat_desc: one product of a syn_mul_mat_batch group."""
    _fields_ = [("type", ctypes.c_int), ("W", ctypes.c_void_p), ("n_out", ctypes.c_int64),
                ("n_in", ctypes.c_int64), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


EXPORTS.append(("syn_mul_mat_batch", _i32, [_i32, ctypes.POINTER(MatDesc), _i64, _vp]))

for _name, _res, _args in EXPORTS:
    _f = getattr(_L, _name)
    _f.restype = _res
    _f.argtypes = _args
    globals()[_name] = _f


class SynError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {syn_strerror(status).decode()} ({status})")
        self.status = status


def check(status: int, what: str = "syn") -> None:
    if status != OK:
        raise SynError(status, what)


# ----------------------------------------------------------------------------------------
# torch-tensor helpers (outputs allocated by torch, work on torch's current stream)
# ----------------------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int:
    return int(t.data_ptr())


def row_bytes(t: int, n: int) -> int:
    return int(syn_row_bytes(t, n))


def quantize(t: int, x, stream=None):
    """fp32 CUDA tensor (n_rows, n) -> uint8 tensor (n_rows, row_bytes)."""
    torch = _torch()
    x = x.contiguous()
    n_rows, n = (1, x.numel()) if x.dim() == 1 else x.shape
    out = torch.empty((n_rows, max(row_bytes(t, n), 0)), dtype=torch.uint8, device=x.device)
    check(syn_quantize(t, _ptr(x), _ptr(out), n_rows, n, _stream(stream)), "syn_quantize")
    return out


def dequantize(t: int, q, n: int, stream=None):
    torch = _torch()
    n_rows = q.numel() // row_bytes(t, n)
    out = torch.empty((n_rows, n), dtype=torch.float32, device=q.device)
    check(syn_dequantize(t, _ptr(q), _ptr(out), n_rows, n, _stream(stream)), "syn_dequantize")
    return out


def quantize_activations(wtype: int, x, stream=None):
    """(qs int8 (n_tok, n_in), d fp32 (n_tok, n_in/Bx), bsums int16 (n_tok, n_in/16) or None)."""
    torch = _torch()
    x = x.contiguous()
    n_tok, n_in = x.shape
    xt = VEC_DOT_TYPE[wtype]
    qs = torch.empty((n_tok, n_in), dtype=torch.int8, device=x.device)
    d = torch.empty((n_tok, n_in // BLOCK_ELEMS[xt]), dtype=torch.float32, device=x.device)
    bs = torch.empty((n_tok, n_in // 16), dtype=torch.int16, device=x.device) if xt == Q8_K else None
    check(syn_quantize_activations(wtype, _ptr(x), n_tok, n_in, _ptr(qs), _ptr(d),
                                   _ptr(bs) if bs is not None else None, _stream(stream)),
          "syn_quantize_activations")
    return qs, d, bs


def mul_mat(t: int, W, n_out: int, n_in: int, X, Y=None, stream=None):
    """Y (n_tok, n_out) fp32 = ggml_mul_mat(W, X); W uint8 blocks, X fp32 (n_tok, n_in)."""
    torch = _torch()
    X = X.contiguous()
    if X.dim() == 1:
        X = X.view(1, -1)
    n_tok = X.shape[0]
    if Y is None:
        Y = torch.empty((n_tok, n_out), dtype=torch.float32, device=X.device)
    check(syn_mul_mat(t, _ptr(W), n_out, n_in, _ptr(X), n_tok, _ptr(Y), _stream(stream)), "syn_mul_mat")
    return Y


def mul_mat_batch(items, n_tok: int, stream=None):
    """items: list of (type, W, n_out, n_in, X, Y) with torch CUDA tensors; one grouped call."""
    arr = (MatDesc * len(items))()
    for k, (t, W, n_out, n_in, X, Y) in enumerate(items):
        arr[k] = MatDesc(t, _ptr(W), n_out, n_in, _ptr(X), _ptr(Y))
    check(syn_mul_mat_batch(len(items), arr, n_tok, _stream(stream)), "syn_mul_mat_batch")


def block_sums(t: int, W, n_out: int, n_in: int, Xq, n_tok: int, stream=None):
    torch = _torch()
    nb = n_in // BLOCK_ELEMS[t]
    S = torch.empty((n_tok, n_out, nb, 2), dtype=torch.int32, device=W.device)
    check(syn_block_sums(t, _ptr(W), n_out, n_in, _ptr(Xq), n_tok, _ptr(S), _stream(stream)), "syn_block_sums")
    return S


def set_gemv_max_tok(n: int) -> int:
    return int(syn_set_gemv_max_tok(n))


def device_status(clear: bool = True) -> int:
    return int(syn_device_status(1 if clear else 0))


def launch_count() -> int:
    return int(syn_launch_count())
