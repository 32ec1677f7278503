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
ERR_FORMAT, ERR_IO, ERR_NOTFOUND = -11, -12, -13
ERR_BOUNDS = -14
# GGUF metadata value types and ggml tensor element types (include/syn.h)
GGUF_UINT8, GGUF_INT8, GGUF_UINT16, GGUF_INT16, GGUF_UINT32, GGUF_INT32, GGUF_FLOAT32, GGUF_BOOL, \
    GGUF_STRING, GGUF_ARRAY, GGUF_UINT64, GGUF_INT64, GGUF_FLOAT64 = range(13)
GGML_F32, GGML_F16, GGML_Q4_0, GGML_Q5_0, GGML_Q8_0, GGML_Q4_K, GGML_Q6_K, GGML_Q8_K, GGML_BF16 = \
    0, 1, 2, 6, 8, 12, 14, 15, 30
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
    ("syn_dequantize_f16", _i32, [_i32, _vp, _vp, _i64, _i64, _vp]),
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
    ("syn_set_deterministic", _i32, [_i32]),
    ("syn_set_sm_limit", _i32, [_i32]),
    ("syn_set_prefill_expand_tok", _i32, [_i32]),
    ("syn_debug_prefill_plan", _i32, [_i64, _i64, _i64, _i32, ctypes.POINTER(ctypes.c_int)]),
    ("syn_debug_bounds_selftest", _i32, [_vp]),
]

class MatDesc(ctypes.Structure):
    """syn_mat_desc: one product of a syn_mul_mat_batch group."""
    _fields_ = [("type", ctypes.c_int), ("W", ctypes.c_void_p), ("n_out", ctypes.c_int64),
                ("n_in", ctypes.c_int64), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


EXPORTS.append(("syn_mul_mat_batch", _i32, [_i32, ctypes.POINTER(MatDesc), _i64, _vp]))
EXPORTS.append(("syn_mul_mat_batch_staged", _i32, [_i32, ctypes.POINTER(MatDesc), _i64, _vp, _vp, ctypes.c_size_t,
                                                   _vp, _vp, ctypes.c_size_t, _vp]))

_u32, _u64, _cp = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_char_p
_P = ctypes.POINTER
EXPORTS += [
    ("syn_gguf_open", _vp, [_cp, _P(_i32)]),
    ("syn_gguf_close", None, [_vp]),
    ("syn_gguf_version", _i64, [_vp]),
    ("syn_gguf_n_tensors", _i64, [_vp]),
    ("syn_gguf_n_kv", _i64, [_vp]),
    ("syn_gguf_alignment", _i64, [_vp]),
    ("syn_gguf_data_start", _i64, [_vp]),
    ("syn_gguf_find_tensor", _i64, [_vp, _cp]),
    ("syn_gguf_tensor_info", _i32, [_vp, _i64, _P(_cp), _P(_u32), _P(_i32), _P(_i64), _P(_u64), _P(_vp),
                                    _P(_i64)]),
    ("syn_gguf_matrix", _i32, [_vp, _cp, _P(_i32), _P(_i64), _P(_i64), _P(_vp), _P(_i64)]),
    ("syn_gguf_upload", _i32, [_vp, _i64, _vp, _i64, _vp]),
    ("syn_gguf_kv_info", _i32, [_vp, _i64, _P(_cp), _P(_u32), _P(_u32), _P(_u64)]),
    ("syn_gguf_get_int", _i32, [_vp, _cp, _P(_i64)]),
    ("syn_gguf_get_float", _i32, [_vp, _cp, _P(ctypes.c_double)]),
    ("syn_gguf_get_string", _i32, [_vp, _cp, _P(_vp), _P(_i64)]),
    ("syn_gguf_get_array", _i32, [_vp, _cp, _P(_u32), _P(_u64), _P(_vp)]),
    ("syn_gguf_get_array_string", _i32, [_vp, _cp, _u64, _P(_vp), _P(_i64)]),
    ("syn_gguf_writer_begin", _vp, [_cp, _u32]),
    ("syn_gguf_writer_kv_int", _i32, [_vp, _cp, _u32, _i64]),
    ("syn_gguf_writer_kv_float", _i32, [_vp, _cp, _u32, ctypes.c_double]),
    ("syn_gguf_writer_kv_string", _i32, [_vp, _cp, _cp, _i64]),
    ("syn_gguf_writer_kv_array", _i32, [_vp, _cp, _u32, _u64, _vp]),
    ("syn_gguf_writer_kv_string_array", _i32, [_vp, _cp, _u64, _P(_cp), _P(_i64)]),
    ("syn_gguf_writer_add_tensor", _i32, [_vp, _cp, _u32, _i32, _P(_i64), _vp, _i64]),
    ("syn_gguf_writer_finish", _i32, [_vp]),
    ("syn_gguf_writer_abort", None, [_vp]),
]

for _name, _res, _args in EXPORTS:
    _f = getattr(_L, _name)
    _f.restype = _res
    _f.argtypes = _args
    globals()[_name] = _f


def bind(path: str):
    """The entry points of another build of the library (a checking variant made by
    ``build.build(variant=...)``) as attributes of a namespace, with the argument types above.
    The helpers below always call libsyn.so."""
    import types
    lib = ctypes.CDLL(path)
    ns = types.SimpleNamespace(path=path)
    for name, res, args in EXPORTS:
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
        setattr(ns, name, f)
    return ns


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
    """A torch stream (None: the current one) or a raw cudaStream_t value, as an integer."""
    if isinstance(stream, int):
        return stream
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


def dequantize_f16(t: int, q, n: int, stream=None):
    """Q4_K / Q6_K blocks -> float16 tensor (n_rows, n): syn_dequantize's values rounded to fp16."""
    torch = _torch()
    n_rows = q.numel() // row_bytes(t, n)
    out = torch.empty((n_rows, n), dtype=torch.float16, device=q.device)
    check(syn_dequantize_f16(t, _ptr(q), _ptr(out), n_rows, n, _stream(stream)), "syn_dequantize_f16")
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


def _descs(items):
    arr = (MatDesc * len(items))()
    for k, (t, W, n_out, n_in, X, Y) in enumerate(items):
        arr[k] = MatDesc(t, _ptr(W), n_out, n_in, _ptr(X), _ptr(Y))
    return arr


def mul_mat_batch(items, n_tok: int, stream=None):
    """items: list of (type, W, n_out, n_in, X, Y) with torch CUDA tensors; one grouped call."""
    check(syn_mul_mat_batch(len(items), _descs(items), n_tok, _stream(stream)), "syn_mul_mat_batch")


class PreparedBatch:
    """A grouped call whose arguments stay the same from call to call (a decode loop over fixed
    buffers): the descriptor array and the stream handle are marshalled once, and each call is
    the one syn_mul_mat_batch call.  With `staged=(x_host, x_dev, y_dev, y_host)` (pinned host
    tensors and the device tensors the products read and write) each call is one
    syn_mul_mat_batch_staged call instead: host-to-device copy, products, device-to-host copy.
    Holds references to the tensors it points at."""

    def __init__(self, items, n_tok: int, stream=None, staged=None):
        self._items = list(items)
        self._arr = _descs(self._items)
        self._n = len(self._items)
        self._n_tok = n_tok
        self._stream = _stream(stream)
        self._staged = staged
        if staged is not None:
            xh, xd, yd, yh = staged
            xb, yb = xh.numel() * xh.element_size(), yh.numel() * yh.element_size()
            if xd.numel() * xd.element_size() < xb or yd.numel() * yd.element_size() < yb:
                raise ValueError("staging buffers smaller than their host counterparts")
            self._sargs = (_ptr(xh), _ptr(xd), xb, _ptr(yd), _ptr(yh), yb)

    def __call__(self):
        if self._staged is None:
            rc = syn_mul_mat_batch(self._n, self._arr, self._n_tok, self._stream)
        else:
            xh, xd, xb, yd, yh, yb = self._sargs
            rc = syn_mul_mat_batch_staged(self._n, self._arr, self._n_tok, xh, xd, xb, yd, yh, yb, self._stream)
        if rc:
            check(rc, "syn_mul_mat_batch")


def prepare_batch(items, n_tok: int, stream=None, staged=None) -> PreparedBatch:
    return PreparedBatch(items, n_tok, stream, staged)


def block_sums(t: int, W, n_out: int, n_in: int, Xq, n_tok: int, stream=None):
    torch = _torch()
    nb = n_in // BLOCK_ELEMS[t]
    S = torch.empty((n_tok, n_out, nb, 2), dtype=torch.int32, device=W.device)
    check(syn_block_sums(t, _ptr(W), n_out, n_in, _ptr(Xq), n_tok, _ptr(S), _stream(stream)), "syn_block_sums")
    return S


def set_gemv_max_tok(n: int) -> int:
    return int(syn_set_gemv_max_tok(n))


def set_deterministic(on: bool) -> bool:
    """Deterministic mode on/off; returns the previous setting."""
    return bool(syn_set_deterministic(1 if on else 0))


def set_prefill_expand_tok(n: int) -> int:
    """Prefill calls of at least n tokens expand K-quant weights to fp16 first (n < 0: the
    default); returns the previous value."""
    return int(syn_set_prefill_expand_tok(n))


def set_sm_limit(n: int) -> int:
    """At most n SMs for the library's launches (0: all); returns the previous limit."""
    return int(syn_set_sm_limit(n))


def device_status(clear: bool = True) -> int:
    return int(syn_device_status(1 if clear else 0))


def launch_count() -> int:
    return int(syn_launch_count())


# ----------------------------------------------------------------------------------------
# GGUF helpers (host side; the tensors come back as numpy views of the mapping)
# ----------------------------------------------------------------------------------------

class GGUFReader:
    """An open GGUF file (syn_gguf_open); ``close()`` unmaps it and invalidates every view."""

    def __init__(self, path: str):
        st = ctypes.c_int(0)
        self.h = syn_gguf_open(os.fsencode(path), ctypes.byref(st))
        if not self.h:
            raise SynError(st.value, f"syn_gguf_open({path})")

    def close(self) -> None:
        if self.h:
            syn_gguf_close(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    version = property(lambda self: int(syn_gguf_version(self.h)))
    alignment = property(lambda self: int(syn_gguf_alignment(self.h)))
    data_start = property(lambda self: int(syn_gguf_data_start(self.h)))
    n_tensors = property(lambda self: int(syn_gguf_n_tensors(self.h)))
    n_kv = property(lambda self: int(syn_gguf_n_kv(self.h)))

    def tensor(self, i: int) -> dict:
        """name, ggml type, ne (n_dims values), offset, nbytes and a uint8 numpy view (or None)."""
        import numpy as np
        name, gt, nd = _cp(), _u32(), _i32()
        ne, off, data, nb = (_i64 * 4)(), _u64(), _vp(), _i64()
        check(syn_gguf_tensor_info(self.h, i, ctypes.byref(name), ctypes.byref(gt), ctypes.byref(nd), ne,
                                   ctypes.byref(off), ctypes.byref(data), ctypes.byref(nb)), "syn_gguf_tensor_info")
        view = None
        if nb.value >= 0:
            view = np.ctypeslib.as_array((ctypes.c_uint8 * nb.value).from_address(data.value)) if nb.value else \
                np.zeros(0, np.uint8)
        return {"name": name.value.decode(), "ggml_type": gt.value, "ne": list(ne[:nd.value]),
                "offset": off.value, "nbytes": nb.value, "data": view}

    def find(self, name: str) -> int:
        return int(syn_gguf_find_tensor(self.h, name.encode()))

    def matrix(self, name: str):
        """(syn type, n_out, n_in, host address, nbytes) of a mul_mat weight."""
        t, n_out, n_in, data, nb = _i32(), _i64(), _i64(), _vp(), _i64()
        check(syn_gguf_matrix(self.h, name.encode(), ctypes.byref(t), ctypes.byref(n_out), ctypes.byref(n_in),
                              ctypes.byref(data), ctypes.byref(nb)), f"syn_gguf_matrix({name})")
        return t.value, n_out.value, n_in.value, data.value, nb.value

    def upload(self, name: str, stream=None):
        """The tensor's bytes copied into a new uint8 CUDA tensor (syn_gguf_upload)."""
        torch = _torch()
        i = self.find(name)
        if i < 0:
            raise SynError(ERR_NOTFOUND, f"syn_gguf_upload({name})")
        nb = self.tensor(i)["nbytes"]
        if nb < 0:
            raise SynError(ERR_TYPE, f"syn_gguf_upload({name})")
        dst = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
        check(syn_gguf_upload(self.h, i, _ptr(dst), dst.numel(), _stream(stream)), f"syn_gguf_upload({name})")
        return dst[:nb]

    def kv_info(self, i: int):
        key, vt, et, n = _cp(), _u32(), _u32(), _u64()
        check(syn_gguf_kv_info(self.h, i, ctypes.byref(key), ctypes.byref(vt), ctypes.byref(et), ctypes.byref(n)),
              "syn_gguf_kv_info")
        return key.value.decode(), vt.value, et.value, n.value

    def get_int(self, key: str) -> int:
        v = _i64()
        check(syn_gguf_get_int(self.h, key.encode(), ctypes.byref(v)), f"syn_gguf_get_int({key})")
        return v.value

    def get_float(self, key: str) -> float:
        v = ctypes.c_double()
        check(syn_gguf_get_float(self.h, key.encode(), ctypes.byref(v)), f"syn_gguf_get_float({key})")
        return v.value

    def get_string(self, key: str) -> bytes:
        p, n = _vp(), _i64()
        check(syn_gguf_get_string(self.h, key.encode(), ctypes.byref(p), ctypes.byref(n)), f"syn_gguf_get_string({key})")
        return ctypes.string_at(p.value, n.value) if n.value else b""

    def get_array(self, key: str):
        """(element type, count, raw little-endian bytes) of a scalar array."""
        et, n, p = _u32(), _u64(), _vp()
        check(syn_gguf_get_array(self.h, key.encode(), ctypes.byref(et), ctypes.byref(n), ctypes.byref(p)),
              f"syn_gguf_get_array({key})")
        return et.value, n.value, p.value

    def get_array_string(self, key: str, j: int) -> bytes:
        p, n = _vp(), _i64()
        check(syn_gguf_get_array_string(self.h, key.encode(), j, ctypes.byref(p), ctypes.byref(n)),
              f"syn_gguf_get_array_string({key}, {j})")
        return ctypes.string_at(p.value, n.value) if n.value else b""


class GGUFWriter:
    """syn_gguf_writer_*: entries are written in call order by ``finish()``."""

    def __init__(self, path: str, alignment: int = 32):
        self.h = syn_gguf_writer_begin(os.fsencode(path), alignment)
        if not self.h:
            raise SynError(ERR_SHAPE, f"syn_gguf_writer_begin({path}, {alignment})")

    def kv_int(self, key: str, value_type: int, value: int) -> None:
        check(syn_gguf_writer_kv_int(self.h, key.encode(), value_type, value), f"kv_int({key})")

    def kv_float(self, key: str, value_type: int, value: float) -> None:
        check(syn_gguf_writer_kv_float(self.h, key.encode(), value_type, value), f"kv_float({key})")

    def kv_string(self, key: str, value: bytes) -> None:
        check(syn_gguf_writer_kv_string(self.h, key.encode(), value, len(value)), f"kv_string({key})")

    def kv_array(self, key: str, elem_type: int, values) -> None:
        """values: a numpy array of the element type's width (its bytes are written as they are)."""
        import numpy as np
        a = np.ascontiguousarray(values)
        check(syn_gguf_writer_kv_array(self.h, key.encode(), elem_type, a.size, a.ctypes.data if a.size else None),
              f"kv_array({key})")

    def kv_string_array(self, key: str, values) -> None:
        n = len(values)
        strs = (_cp * max(n, 1))(*values)
        lens = (_i64 * max(n, 1))(*[len(v) for v in values])
        check(syn_gguf_writer_kv_string_array(self.h, key.encode(), n, strs, lens), f"kv_string_array({key})")

    def add_tensor(self, name: str, ggml_type: int, ne, data) -> None:
        """data: a numpy array holding the tensor's bytes (any dtype, C-contiguous)."""
        import numpy as np
        a = np.ascontiguousarray(data)
        arr = (_i64 * len(ne))(*ne)
        check(syn_gguf_writer_add_tensor(self.h, name.encode(), ggml_type, len(ne), arr,
                                         a.ctypes.data if a.nbytes else None, a.nbytes), f"add_tensor({name})")

    def finish(self) -> None:
        h, self.h = self.h, None
        check(syn_gguf_writer_finish(h), "syn_gguf_writer_finish")

    def abort(self) -> None:
        if self.h:
            syn_gguf_writer_abort(self.h)
            self.h = None
