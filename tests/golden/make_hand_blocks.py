"""Writes hand_blocks.txt: one hand-made block per format, as raw bytes plus its fields.

The bytes are test INPUTS.  They are packed here from chosen field values, bit by bit,
following the in-block layout the library and the oracle both use (the public GGUF
layout).  This script does not call the oracle or the library; the tests decode the bytes
with the oracle and compare against the format formulas of "The GGML ecosystem, and
where synapse fits", section 5 (Q8_0: w = d*q; Q4_K: w = d*sc*q - dmin*m;
Q6_K: w = d*sc*(q - 32); Q8_K: w = d*q with bsums = sums of 16 codes; Q4_0: w = d*(q - 8);
Q5_0: w = d*(q - 16) with the fifth bits in a 32-bit qh).

Run: python tests/golden/make_hand_blocks.py   (rewrites hand_blocks.txt beside it)
"""
import os
import struct


def bits_set(buf, bit_offset, value, nbits):
    """Write `value` (nbits wide) into byte buffer `buf` starting at an absolute bit."""
    for k in range(nbits):
        if (value >> k) & 1:
            buf[(bit_offset + k) // 8] |= 1 << ((bit_offset + k) % 8)


def q4_k_block():
    d, dmin = 0x3C00, 0x3800  # fp16 1.0 and 0.5
    sc = [1, 2, 3, 4, 17, 33, 47, 63]
    mn = [0, 1, 2, 3, 20, 35, 50, 62]
    q = [((i % 32) + (i // 32)) % 16 for i in range(256)]  # sub-block j element l -> (l + j) % 16
    buf = bytearray(144)
    buf[0:2] = struct.pack("<H", d)
    buf[2:4] = struct.pack("<H", dmin)
    base = 4 * 8
    for j in range(4):
        bits_set(buf, base + 8 * j, sc[j], 6)                    # byte j, bits 0-5
        bits_set(buf, base + 8 * j + 6, sc[j + 4] >> 4, 2)       # byte j, bits 6-7
        bits_set(buf, base + 8 * (j + 4), mn[j], 6)              # byte j+4, bits 0-5
        bits_set(buf, base + 8 * (j + 4) + 6, mn[j + 4] >> 4, 2) # byte j+4, bits 6-7
        bits_set(buf, base + 8 * (j + 8), sc[j + 4] & 15, 4)     # byte j+8, low nibble
        bits_set(buf, base + 8 * (j + 8) + 4, mn[j + 4] & 15, 4) # byte j+8, high nibble
    for i in range(256):
        chunk, within = divmod(i, 64)          # 64 weights per 32-byte chunk
        high, l = divmod(within, 32)           # first 32 -> low nibbles, next 32 -> high
        bits_set(buf, 8 * (16 + 32 * chunk + l) + 4 * high, q[i], 4)
    return bytes(buf), dict(d=d, dmin=dmin, sc=sc, mn=mn, q=q)


def q6_k_block():
    d = 0x3400  # fp16 0.25
    sc = [8 * j - 60 for j in range(16)]  # includes negative int8 scales
    q = [(7 * i + 3) % 64 for i in range(256)]
    buf = bytearray(210)
    for i in range(256):
        h, w = divmod(i, 128)                 # half, weight within the half
        quarter, l = divmod(w, 32)            # weights l, l+32, l+64, l+96
        ql_byte = 64 * h + l + (32 if quarter in (1, 3) else 0)
        ql_shift = 4 if quarter in (2, 3) else 0
        bits_set(buf, 8 * ql_byte + ql_shift, q[i] & 15, 4)
        bits_set(buf, 8 * (128 + 32 * h + l) + 2 * quarter, q[i] >> 4, 2)
    for j in range(16):
        buf[192 + j] = sc[j] & 0xFF
    buf[208:210] = struct.pack("<H", d)
    return bytes(buf), dict(d=d, sc=sc, q=q)


def q8_0_block():
    d = 0x2C08  # fp16 129/2048
    q = [((5 * i) % 255) - 127 for i in range(32)]
    buf = bytearray(34)
    buf[0:2] = struct.pack("<H", d)
    for i in range(32):
        buf[2 + i] = q[i] & 0xFF
    return bytes(buf), dict(d=d, q=q)


def q8_k_block():
    d = 0.125
    q = [(i % 255) - 127 if i % 3 else 127 - (i % 200) for i in range(256)]
    bsums = [sum(q[16 * k:16 * k + 16]) for k in range(16)]
    buf = bytearray(292)
    buf[0:4] = struct.pack("<f", d)
    for i in range(256):
        buf[4 + i] = q[i] & 0xFF
    for k in range(16):
        buf[260 + 2 * k:262 + 2 * k] = struct.pack("<h", bsums[k])
    return bytes(buf), dict(d=d, q=q, bsums=bsums)


def q4_0_block():
    d = 0x3A00  # fp16 0.75
    q = [(3 * i + 1) % 16 for i in range(32)]
    buf = bytearray(18)
    buf[0:2] = struct.pack("<H", d)
    for i in range(32):
        l, high = i % 16, i // 16              # weights l (low nibble) and l + 16 (high)
        bits_set(buf, 8 * (2 + l) + 4 * high, q[i], 4)
    return bytes(buf), dict(d=d, q=q)


def q5_0_block():
    d = 0x3100  # fp16 0.15625
    q = [(7 * i + 5) % 32 for i in range(32)]
    buf = bytearray(22)
    buf[0:2] = struct.pack("<H", d)
    for i in range(32):
        bits_set(buf, 8 * 2 + i, q[i] >> 4, 1)  # qh: bit i of a little-endian 32-bit word
        l, high = i % 16, i // 16
        bits_set(buf, 8 * (6 + l) + 4 * high, q[i] & 15, 4)
    return bytes(buf), dict(d=d, q=q)


def main():
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "hand_blocks.txt")
    lines = ["# Hand-made blocks (inputs) written by make_hand_blocks.py; fields then hex bytes.",
             "# Formulas checked by the tests: format table of 'The GGML ecosystem, and where",
             "# synapse fits', section 5."]
    for name, (raw, f) in [("Q8_0", q8_0_block()), ("Q4_K", q4_k_block()),
                           ("Q6_K", q6_k_block()), ("Q8_K", q8_k_block()),
                           ("Q4_0", q4_0_block()), ("Q5_0", q5_0_block())]:
        lines.append(f"[{name}]")
        for k, v in f.items():
            lines.append(f"{k} = {' '.join(map(str, v)) if isinstance(v, list) else v}")
        lines.append("hex = " + raw.hex())
    with open(out, "w") as fh:
        fh.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
