"""GGUF container layout in plain Python — TEST INFRASTRUCTURE ONLY.

Only the tests may import this module; the library never does, and it shares no code with
the library's reader and writer (``csrc/gguf.cpp``).  It writes and reads the layout field
by field with ``struct``, in the order the pages give:

  "The GGML ecosystem, and where synapse fits", section 2 (the GGUF diagram and the tensor
  info bullets: ne innermost first, ne = [cols, rows] for a weight matrix);
  "ggml Documentation", GGUF specification, "File Structure" (global alignment, zero
  padding, fields packed without alignment, little-endian) and the general.alignment key
  (uint32, a multiple of 8, 32 when absent);
  "llama.cpp and GGUF", "GGUF: The Single-File Container" (header: magic, version,
  tensor_count, kv_count; metadata; tensor infos; aligned data).

Readings where the pages leave a detail open (each also used, independently, by the library):
  * counts, lengths, dimensions and offsets are u64, the version, value types, n_dims and
    tensor types u32 (the diagram's widths; the rest from the public GGUF specification);
  * a string is its u64 byte count followed by the bytes; an array is element type u32,
    count u64, the elements;
  * a tensor's offset counts from the start of the data section (the first multiple of the
    alignment after the tensor infos).  "llama.cpp and GGUF" calls the offsets absolute; the
    ggml-ecosystem diagram places each tensor "at its offset" inside the data section.  The
    two readings differ; this one is the public specification's;
  * numeric codes of value types and tensor types: the public GGUF specification.

Parity status: pinned to hand-assembled byte strings (tests/golden/gguf_tiny.txt) and to
hand-computed offsets; the numeric codes above are unpinned readings (no real GGUF file is
available to check them against).
"""
from __future__ import annotations

import struct

MAGIC = b"GGUF"
DEFAULT_ALIGNMENT = 32

# metadata value types
UINT8, INT8, UINT16, INT16, UINT32, INT32, FLOAT32, BOOL, STRING, ARRAY, UINT64, INT64, FLOAT64 = range(13)
_SCALAR = {UINT8: "<B", INT8: "<b", UINT16: "<H", INT16: "<h", UINT32: "<I", INT32: "<i", FLOAT32: "<f",
           BOOL: "<?", UINT64: "<Q", INT64: "<q", FLOAT64: "<d"}

# ggml tensor element types: code -> (name, elements per block, bytes per block)
GGML_TYPES = {
    0: ("F32", 1, 4),
    1: ("F16", 1, 2),
    2: ("Q4_0", 32, 18),
    6: ("Q5_0", 32, 22),
    8: ("Q8_0", 32, 34),
    12: ("Q4_K", 256, 144),
    14: ("Q6_K", 256, 210),
    15: ("Q8_K", 256, 292),
    30: ("BF16", 1, 2),
}
GGML_CODE = {name: code for code, (name, _, _) in GGML_TYPES.items()}


def _pad_to(n: int, a: int) -> int:
    return (n + a - 1) // a * a


def _string(b: bytes) -> bytes:
    return struct.pack("<Q", len(b)) + b


def _value(vtype: int, value) -> bytes:
    if vtype == STRING:
        return _string(value)
    if vtype == ARRAY:
        etype, items = value
        out = struct.pack("<IQ", etype, len(items))
        for it in items:
            out += _value(etype, it)
        return out
    return struct.pack(_SCALAR[vtype], value)


def serialize(kv, tensors, alignment: int = DEFAULT_ALIGNMENT) -> bytes:
    """A version-3 GGUF file.

    kv: list of (key: bytes, value type, value): scalars as Python numbers, strings as bytes,
        arrays as (element type, list of values).  A general.alignment entry, if the file
        should carry one, is part of this list like any other.
    tensors: list of (name: bytes, ggml type code, ne list innermost first, data: bytes);
        each is placed at the next multiple of ``alignment`` in the data section.
    """
    head = MAGIC + struct.pack("<IQQ", 3, len(tensors), len(kv))
    meta = b"".join(_string(k) + struct.pack("<I", t) + _value(t, v) for k, t, v in kv)
    info, data = b"", b""
    for name, gtype, ne, blob in tensors:
        off = _pad_to(len(data), alignment)
        data += b"\0" * (off - len(data)) + blob
        info += _string(name) + struct.pack("<I", len(ne)) + b"".join(struct.pack("<Q", d) for d in ne)
        info += struct.pack("<IQ", gtype, off)
    pre = head + meta + info
    return pre + b"\0" * (_pad_to(len(pre), alignment) - len(pre)) + data


class _In:
    def __init__(self, buf: bytes):
        self.buf, self.at = buf, 0

    def take(self, fmt: str):
        v = struct.unpack_from(fmt, self.buf, self.at)[0]
        self.at += struct.calcsize(fmt)
        return v

    def string(self) -> bytes:
        n = self.take("<Q")
        if self.at + n > len(self.buf):
            raise ValueError("string past the end of the file")
        s = self.buf[self.at:self.at + n]
        self.at += n
        return s

    def value(self, vtype: int):
        if vtype == STRING:
            return self.string()
        if vtype == ARRAY:
            etype = self.take("<I")
            n = self.take("<Q")
            return (etype, [self.value(etype) for _ in range(n)])
        if vtype not in _SCALAR:
            raise ValueError(f"unknown value type {vtype}")
        return self.take(_SCALAR[vtype])


def parse(buf: bytes) -> dict:
    """The fields of a GGUF file: version, kv (list of (key, type, value)), alignment,
    tensors (list of dicts: name, ne, type, offset), data_start.  Raises ValueError (or
    struct.error past the end) on a malformed file."""
    if buf[:4] != MAGIC:
        raise ValueError("bad magic")
    r = _In(buf)
    r.at = 4
    version = r.take("<I")
    n_tensors = r.take("<Q")
    n_kv = r.take("<Q")
    kv = []
    alignment = DEFAULT_ALIGNMENT
    for _ in range(n_kv):
        key = r.string()
        vtype = r.take("<I")
        val = r.value(vtype)
        kv.append((key, vtype, val))
        if key == b"general.alignment":
            if vtype != UINT32 or val == 0 or val % 8:
                raise ValueError("general.alignment must be a uint32 multiple of 8")
            alignment = val
    tensors = []
    for _ in range(n_tensors):
        name = r.string()
        n_dims = r.take("<I")
        ne = [r.take("<Q") for _ in range(n_dims)]
        gtype = r.take("<I")
        offset = r.take("<Q")
        tensors.append({"name": name, "ne": ne, "type": gtype, "offset": offset})
    return {"version": version, "kv": kv, "alignment": alignment, "tensors": tensors,
            "data_start": _pad_to(r.at, alignment)}


def tensor_nbytes(gtype: int, ne) -> int:
    _, elems, nbytes = GGML_TYPES[gtype]
    count = 1
    for d in ne:
        count *= d
    if ne[0] % elems:
        raise ValueError("a row is not a whole number of blocks")
    return count // elems * nbytes


def tensor_bytes(buf: bytes, parsed: dict, name: bytes) -> bytes:
    """The data bytes of tensor ``name`` in a parsed file."""
    for t in parsed["tensors"]:
        if t["name"] == name:
            start = parsed["data_start"] + t["offset"]
            return buf[start:start + tensor_nbytes(t["type"], t["ne"])]
    raise KeyError(name)
