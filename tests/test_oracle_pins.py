"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test names the passage (web page + section) or the mathematical fact it checks.
Runs on CPU only (no GPU marker).
"""
import os
import struct

import numpy as np
import pytest

import oracle
from oracle import Q8_0, Q4_K, Q6_K, Q8_K, Q4_0, Q5_0
from conftest import GOLDEN, read_fixture
from gguf_block_quantized_gb300 import synth, workloads


def f16(bits):
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


# ----------------------------------------------------------------------------------------
# fp32 -> fp16 round-to-nearest-even: pinned to numpy's IEEE conversion
# ----------------------------------------------------------------------------------------

def _numpy_half_bits(x):
    with np.errstate(over="ignore"):
        return x.astype(np.float16).view(np.uint16)


def _compare_half(x):
    mine = oracle.fp32_to_fp16_bits(x)
    ref = _numpy_half_bits(x)
    nan = np.isnan(x)
    assert np.all((mine[nan] & 0x7C00) == 0x7C00) and np.all((mine[nan] & 0x3FF) != 0)
    bad = np.nonzero((mine != ref) & ~nan)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x bits {x.view(np.uint32)[bad[:4]]}"


def test_fp16_rne_every_boundary():
    """Every fp16 value h, every midpoint between neighbours, and +-1 ulp around each."""
    h = np.arange(0, 0x7C00, dtype=np.uint32)  # all finite non-negative fp16 values
    vals = np.array(h, dtype=np.uint16).view(np.float16).astype(np.float64)
    nxt = np.append(vals[1:], 65536.0)
    mid = ((vals + nxt) / 2).astype(np.float32)  # exact in fp32
    base = np.concatenate([vals.astype(np.float32), mid])
    u = base.view(np.uint32)
    cand = np.concatenate([u, u + 1, u - 1, u + 7, u - 7]).astype(np.uint32)
    cand = cand[(cand & 0x7F800000) != 0x7F800000]
    x = cand.view(np.float32)
    _compare_half(np.concatenate([x, -x]))


def test_fp16_rne_dense_sample_all_exponents():
    rng = np.random.default_rng(7)
    u = rng.integers(0, 2**32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 65504, 65519.996, 65520, 65536,
                         2.0**-24, 2.0**-25, 2.0**-25 * 1.0000001, 2.0**-14, 1e-45, 3e38],
                        dtype=np.float32)
    _compare_half(np.concatenate([x, specials, -specials]))


def test_fp16_to_fp32_exact_all_values():
    h = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    mine = oracle.fp16_bits_to_fp32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.all(np.isnan(mine[nan]))
    assert np.array_equal(mine[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ----------------------------------------------------------------------------------------
# block sizes (format table) and bits per weight
# ----------------------------------------------------------------------------------------

def test_block_sizes_match_format_table():
    # "The GGML ecosystem, and where synapse fits", section 5, format table.
    L = oracle.lib()
    assert [L.orc_block_elems(t) for t in (Q8_0, Q4_K, Q6_K, Q8_K, Q4_0, Q5_0)] == [32, 256, 256, 256, 32, 32]
    assert [L.orc_block_bytes(t) for t in (Q8_0, Q4_K, Q6_K, Q8_K, Q4_0, Q5_0)] == [34, 144, 210, 292, 18, 22]
    # Q4_0: fp16 d + 32 x 4 bits; Q5_0: fp16 d + 32-bit qh + 32 x 4 bits
    assert 2 + 32 * 4 // 8 == 18 and 2 + 4 + 32 * 4 // 8 == 22
    # Q6_K: 256 x 4 bits + 256 x 2 bits + 16 int8 scales + fp16 d
    assert 256 * 4 // 8 + 256 * 2 // 8 + 16 + 2 == 210


def test_bits_per_weight():
    # Q4_K "reaches 4.5 bits per weight" (section 5); Q8_0 "~8.5 bpw" ("llama.cpp and GGUF").
    bpw = {t: 8 * oracle.BLOCK_BYTES[t] / oracle.BLOCK_ELEMS[t] for t in (Q8_0, Q4_K, Q6_K, Q8_K)}
    assert bpw[Q4_K] == 4.5 and bpw[Q8_0] == 8.5
    assert bpw[Q6_K] == 6.5625 and bpw[Q8_K] == 9.125
    # the legacy 32-weight formats span "4.5 - 8.5" bpw ("llama.cpp and GGUF", format table)
    assert 8 * 18 / 32 == 4.5 and 8 * 22 / 32 == 5.5


def test_llama8b_q4_k_m_size_in_published_range():
    """'llama.cpp and GGUF': Llama-3.1-8B Q4_K_M ~4.9 GB; 7-8B sizes Q4_K_M 4.4-4.9 GB,
    Q6_K 6.3-6.6 GB, Q8_0 8.1-8.5 GB.  Token embedding (Q4_K) counted as stored bytes."""
    mats = workloads.llama8b_q4_k_m()
    emb = workloads.Matrix("token_embd", Q4_K, 128256, 4096)
    total = sum(m.weight_bytes for m in mats) + emb.weight_bytes
    assert 4.4e9 <= total <= 4.95e9
    n_w = sum(m.n_out * m.n_in for m in mats) + emb.n_out * emb.n_in
    assert 6.3e9 <= n_w * 6.5625 / 8 <= 6.65e9
    assert 8.1e9 <= n_w * 8.5 / 8 <= 8.6e9
    assert sum(1 for m in mats if m.wtype == Q6_K) == 2 * 16 + 1  # v, down in 16 layers + lm_head


# ----------------------------------------------------------------------------------------
# hand-made blocks against the format formulas (dequantize pins the byte layout reading)
# ----------------------------------------------------------------------------------------

HB = read_fixture(os.path.join(GOLDEN, "hand_blocks.txt"))


def _ints(s):
    return np.array([int(v) for v in s.split()], dtype=np.int64)


def _raw(sec):
    return np.frombuffer(bytes.fromhex(HB[sec]["hex"]), dtype=np.uint8)


def test_hand_q8_0_dequant():
    f = HB["Q8_0"]
    d = f16(int(f["d"]))
    want = (np.float32(d) * _ints(f["q"]).astype(np.float32)).astype(np.float32)
    got = oracle.dequantize(Q8_0, _raw("Q8_0"), 32)[0]
    assert np.array_equal(got, want)


def test_hand_q4_k_dequant_and_fields():
    f = HB["Q4_K"]
    d, dmin = f16(int(f["d"])), f16(int(f["dmin"]))
    sc, mn, q = _ints(f["sc"]), _ints(f["mn"]), _ints(f["q"])
    raw = _raw("Q4_K")
    gd, gdm, gsc, gmn, gq = oracle.unpack_q4_k(raw)
    assert (gd, gdm) == (int(f["d"]), int(f["dmin"]))
    assert list(gsc) == list(sc) and list(gmn) == list(mn) and list(gq) == list(q)
    j = np.arange(256) // 32
    want = d * sc[j] * q - dmin * mn[j]  # exact in fp64 and in fp32 for these values
    got = oracle.dequantize(Q4_K, raw, 256)[0]
    assert np.array_equal(got.astype(np.float64), want)


def test_hand_q6_k_dequant_and_fields():
    f = HB["Q6_K"]
    d = f16(int(f["d"]))
    sc, q = _ints(f["sc"]), _ints(f["q"])
    raw = _raw("Q6_K")
    gd, gsc, gq = oracle.unpack_q6_k(raw)
    assert gd == int(f["d"]) and list(gsc) == list(sc) and list(gq) == list(q)
    want = d * sc[np.arange(256) // 16] * (q - 32)
    got = oracle.dequantize(Q6_K, raw, 256)[0]
    assert np.array_equal(got.astype(np.float64), want)


def test_hand_q8_k_dequant_and_bsums():
    f = HB["Q8_K"]
    raw = _raw("Q8_K")
    d = float(f["d"])
    q = _ints(f["q"])
    got = oracle.dequantize(Q8_K, raw, 256)[0]
    assert np.array_equal(got.astype(np.float64), d * q)
    bs = np.frombuffer(raw[260:292].tobytes(), dtype="<i2")
    assert list(bs) == list(_ints(f["bsums"])) == [int(q[16 * k:16 * k + 16].sum()) for k in range(16)]


@pytest.mark.parametrize("t,off", [(Q4_0, 8), (Q5_0, 16)])
def test_hand_qx_0_dequant_and_fields(t, off):
    name = oracle.NAMES[t]
    f = HB[name]
    d, q = f16(int(f["d"])), _ints(f["q"])
    raw = _raw(name)
    gd, gq = oracle.unpack_qx_0(t, raw)
    assert gd == int(f["d"]) and list(gq) == list(q)
    got = oracle.dequantize(t, raw, 32)[0]
    assert np.array_equal(got.astype(np.float64), d * (q - off))


# ----------------------------------------------------------------------------------------
# Q8_0 worked example and rounding-tie reading
# ----------------------------------------------------------------------------------------

W8 = read_fixture(os.path.join(GOLDEN, "q8_0_worked.txt"))


def test_q8_0_worked_block():
    x = np.array([(i - 16) * 0.5 for i in range(32)], dtype=np.float32)
    b = oracle.quantize(Q8_0, x)[0]
    assert int(b[0]) | (int(b[1]) << 8) == int(W8["d_bits"], 16)
    assert list(b[2:].view(np.int8)) == list(_ints(W8["q"]))


def test_q8_0_ties_away_from_zero():
    tx = np.array([float(v) for v in W8["tie_x"].split()], dtype=np.float32)
    tq = _ints(W8["tie_q"])
    x = np.zeros(32, np.float32)
    x[:tx.size] = tx
    b = oracle.quantize(Q8_0, x)[0]
    assert int(b[0]) | (int(b[1]) << 8) == 0x3C00  # scale exactly 1
    assert list(b[2:2 + tx.size].view(np.int8)) == list(tq)


# ----------------------------------------------------------------------------------------
# K-quant encoders: hand-worked super-blocks (format table, "The GGML ecosystem...", section 5;
# the min-max / symmetric readings of the Q4_K and Q6_K rows).  Scales are chosen so that
# round and floor, and round-half-away and round-half-even, give different sub-block scales,
# and so that the super-scales are powers of two only for the divisors 63 / 127.
# ----------------------------------------------------------------------------------------

WQ4 = read_fixture(os.path.join(GOLDEN, "q4_k_worked.txt"))
WQ6 = read_fixture(os.path.join(GOLDEN, "q6_k_worked.txt"))


def _worked_inputs(fix, n_sub):
    x = np.concatenate([np.array([float(v) for v in fix[f"x{j}"].split()], dtype=np.float32)
                        for j in range(n_sub)])
    assert x.size == 256
    return x


def test_q4_k_worked_block():
    x = _worked_inputs(WQ4, 8)
    b = oracle.quantize(Q4_K, x.reshape(1, 256))[0]
    d, dm, sc, mn, q = oracle.unpack_q4_k(b)
    assert d == int(WQ4["d_bits"], 16) and dm == int(WQ4["dmin_bits"], 16)
    assert [int(v) for v in sc] == list(_ints(WQ4["sc"]))
    assert [int(v) for v in mn] == list(_ints(WQ4["mn"]))
    first, second, lst = _ints(WQ4["q_first"]), _ints(WQ4["q_second"]), _ints(WQ4["q_list"])
    for j in range(8):
        qj = [int(v) for v in q[32 * j:32 * j + 32]]
        want = [0] * 32 if int(_ints(WQ4["sc"])[j]) == 0 else [int(first[j]), int(second[j])] + list(lst)
        assert qj == want, j


def test_q6_k_worked_block():
    x = _worked_inputs(WQ6, 16)
    b = oracle.quantize(Q6_K, x.reshape(1, 256))[0]
    d, sc, q = oracle.unpack_q6_k(b)
    assert d == int(WQ6["d_bits"], 16)
    assert [int(v) for v in sc] == list(_ints(WQ6["sc"]))
    first, lst = _ints(WQ6["q_first"]), _ints(WQ6["q_list"])
    zero = set(int(v) for v in _ints(WQ6["zero_code_subblocks"]))
    for j in range(16):
        qj = [int(v) for v in q[16 * j:16 * j + 16]]
        want = [32] * 16 if j in zero else [int(first[j])] + list(lst)
        assert qj == want, j


def test_zero_blocks_give_zero_scales_and_codes():
    for t in (Q8_0, Q4_K, Q6_K, Q8_K):
        n = oracle.BLOCK_ELEMS[t]
        b = oracle.quantize(t, np.zeros(n, np.float32))
        assert np.array_equal(oracle.dequantize(t, b, n), np.zeros((1, n), np.float32))
        if t == Q6_K:  # codes stored with the +32 offset
            _, sc, q = oracle.unpack_q6_k(b[0])
            assert np.all(sc == 0) and np.all(q == 32)
        elif t == Q4_K:
            d, dm, sc, mn, q = oracle.unpack_q4_k(b[0])
            assert d == 0 and dm == 0 and np.all(q == 0)
        else:
            assert np.count_nonzero(b) == 0


# ----------------------------------------------------------------------------------------
# error bounds of quantize -> dequantize (closed forms from the formulas)
# ----------------------------------------------------------------------------------------

def _test_inputs(n):
    """A mix of distributions, with the degenerate cases the formats have."""
    rows = [
        synth.normal(11, n, 0.02),
        synth.normal(12, n, 1.0),
        synth.uniform(13, n, -3.0, 3.0),
        synth.uniform(14, n, -5.0, -0.5),         # all negative
        synth.uniform(15, n, 0.25, 4.0),          # all positive
        synth.normal(16, n, 1e-6),                # fp16-subnormal scales
        np.full(n, 0.375, np.float32),            # constant
        np.full(n, -2.0, np.float32),
    ]
    spike = synth.normal(17, n, 0.01)
    spike[::37] *= 300.0                          # outliers
    rows.append(spike)
    sparse = synth.normal(18, n, 1.0)
    sparse[synth.integers(19, n, 0, 4) != 0] = 0.0
    rows.append(sparse)
    heavy = synth.normal(20, n, 1.0) ** 3
    rows.append(heavy.astype(np.float32))
    return np.stack(rows).astype(np.float32)


def _ulp_slack(*mags):
    return 4 * np.spacing(np.float32(np.max(np.abs(np.stack(mags)), axis=0)).astype(np.float32))


def test_q8_0_error_bound():
    x = _test_inputs(1024)
    b = oracle.quantize(Q8_0, x)
    y = oracle.dequantize(Q8_0, b, 1024)
    D = np.array([f16(int(b[r, 34 * k]) | (int(b[r, 34 * k + 1]) << 8))
                  for r in range(x.shape[0]) for k in range(32)]).reshape(x.shape[0], 32)
    amax = np.abs(x.reshape(x.shape[0], 32, 32)).max(axis=2)
    # |x - q*D| <= D/2 while amax/D <= 127; when fp16 rounding made D smaller than
    # amax/127 (subnormal range) the +-127 clamp can add amax - 127*D.
    bound = np.maximum(D / 2, amax - 127 * D)
    assert np.all(np.abs(x - y) <= np.repeat(bound, 32, axis=1) + _ulp_slack(x, y))
    normal = D >= 2.0 ** -14
    assert np.all((amax - 127 * D)[normal] <= D[normal] / 2)
    # the stored scale is amax/127 rounded once to fp16
    d = (amax / np.float32(127)).astype(np.float32)
    assert np.array_equal(D.astype(np.float16), d.astype(np.float16).astype(np.float64).astype(np.float16))


def test_q8_k_error_bound_and_bsums():
    x = _test_inputs(1024)
    b = oracle.quantize(Q8_K, x).reshape(x.shape[0], 4, 292)
    y = oracle.dequantize(Q8_K, b, 1024)
    d = b[:, :, 0:4].copy().view(np.float32).reshape(x.shape[0], 4)
    amax = np.abs(x.reshape(x.shape[0], 4, 256)).max(axis=2)
    assert np.array_equal(d, (amax / np.float32(127)).astype(np.float32))
    q = b[:, :, 4:260].view(np.int8).astype(np.int64)
    bs = b[:, :, 260:292].copy().view("<i2").astype(np.int64)
    assert np.array_equal(bs, q.reshape(x.shape[0], 4, 16, 16).sum(axis=3))
    assert np.all(np.abs(q) <= 127)
    assert np.all(np.abs(x - y) <= np.repeat(d, 256, axis=1) / 2 + _ulp_slack(x, y))


def test_q4_k_error_bound():
    x = _test_inputs(1024)
    n_rows = x.shape[0]
    b = oracle.quantize(Q4_K, x).reshape(n_rows, 4, 144)
    y = oracle.dequantize(Q4_K, b, 1024)
    for r in range(n_rows):
        for k in range(4):
            d, dm, sc, mn, q = oracle.unpack_q4_k(b[r, k])
            D, Dm = np.float32(f16(d)), np.float32(f16(dm))
            for j in range(8):
                xs = x[r, 256 * k + 32 * j: 256 * k + 32 * j + 32]
                ys = y[r, 256 * k + 32 * j: 256 * k + 32 * j + 32]
                lo, hi = min(0.0, float(xs.min())), float(xs.max())
                s, m = (hi - lo) / 15.0, -lo
                S, M = float(D) * int(sc[j]), float(Dm) * int(mn[j])
                bound = max(S / 2, abs(m - M) + 15 * abs(s - S))
                slack = 1e-6 * (np.abs(xs).max() + M + 16 * S) + 1e-30
                assert np.all(np.abs(xs - ys) <= bound + slack), (r, k, j)
                assert np.all(q[32 * j:32 * j + 32] <= 15)


def test_q6_k_error_bound():
    x = _test_inputs(1024)
    n_rows = x.shape[0]
    b = oracle.quantize(Q6_K, x).reshape(n_rows, 4, 210)
    y = oracle.dequantize(Q6_K, b, 1024)
    for r in range(n_rows):
        for k in range(4):
            d, sc, q = oracle.unpack_q6_k(b[r, k])
            D = float(np.float32(f16(d)))
            for j in range(16):
                xs = x[r, 256 * k + 16 * j: 256 * k + 16 * j + 16]
                ys = y[r, 256 * k + 16 * j: 256 * k + 16 * j + 16]
                s = float(np.abs(xs).max()) / 31.0
                S = D * int(sc[j])
                bound = max(S / 2, 31 * abs(s - S))
                slack = 1e-6 * (np.abs(xs).max() + 32 * S) + 1e-30
                assert np.all(np.abs(xs - ys) <= bound + slack), (r, k, j)
                assert 0 <= int(sc[j]) <= 127


@pytest.mark.parametrize("t,off", [(Q4_0, 8), (Q5_0, 16)])
def test_qx_0_error_bound_and_extreme(t, off):
    """w = d*(q - off) (format table): with d = m/-off for the block's largest-magnitude value
    m, every weight is within D/2 of its input, except inputs above (off - 1/2)*|D| on the
    side opposite to m, which clip to q = 2*off - 1 (within |D|); m itself is reproduced up
    to the fp16 rounding of d."""
    x = _test_inputs(512)
    y = oracle.dequantize(t, oracle.quantize(t, x), 512)
    b = oracle.quantize(t, x).reshape(x.shape[0], -1, oracle.BLOCK_BYTES[t])
    for r in range(x.shape[0]):
        for k in range(512 // 32):
            xs, ys = x[r, 32 * k:32 * k + 32].astype(np.float64), y[r, 32 * k:32 * k + 32].astype(np.float64)
            D = f16(int(b[r, k, 0]) | int(b[r, k, 1]) << 8)
            i = int(np.argmax(np.abs(xs)))
            m = xs[i]
            if m == 0:
                assert np.all(ys == 0)
                continue
            # fp16 rounding of d = m/-off: half an ulp, 2^-11 relative or 2^-25 absolute
            # (subnormal); m is reproduced up to off times that
            err_d = max(2 ** -11 * abs(m) / off, 2 ** -25)
            slack = 1e-6 * np.abs(xs).max() + 1e-30
            assert abs(ys[i] - m) <= off * err_d + slack
            u = xs / D  # in [-off, off] up to the rounding of D
            clip = u > off - 0.5
            assert np.all(np.abs(xs - ys)[~clip] <= abs(D) / 2 + off * err_d + slack)
            assert np.all(np.abs(xs - ys)[clip] <= abs(D) + off * err_d + slack)


@pytest.mark.parametrize("t", [Q8_0, Q8_K, Q4_0, Q5_0])
def test_requantize_is_a_fixed_point(t):
    """quantize(dequantize(quantize(x))) == quantize(x), byte for byte.

    Holds exactly for the symmetric 8-bit formats: the largest code is +-127, so the
    re-derived scale is 127*D/127 = D and every code divides back exactly; likewise for
    Q4_0/Q5_0, whose largest-magnitude value dequantizes to -off*D.  (The K-quant encoders
    are not idempotent on outlier blocks, so they are pinned by their bounds.)"""
    x = _test_inputs(512)
    b1 = oracle.quantize(t, x)
    b2 = oracle.quantize(t, oracle.dequantize(t, b1, 512))
    assert np.array_equal(b1, b2)


def test_range_errors():
    for t in (Q8_0, Q4_K, Q6_K, Q8_K, Q4_0, Q5_0):
        n = oracle.BLOCK_ELEMS[t]
        for bad in (np.nan, np.inf, -np.inf):
            x = np.zeros(n, np.float32); x[3] = bad
            assert oracle.quantize_status(t, x) == -5
    # a scale that overflows fp16: amax/127 > 65504
    x = np.zeros(32, np.float32); x[0] = 1e7
    assert oracle.quantize_status(Q8_0, x) == -5
    x = np.zeros(256, np.float32); x[0] = 1e9
    assert oracle.quantize_status(Q4_K, x) == -5 and oracle.quantize_status(Q6_K, x) == -5
    assert oracle.quantize_status(Q8_K, x) == 0  # Q8_K keeps d in fp32
    assert oracle.quantize_status(Q4_K, np.zeros(100, np.float32)) == -2


# ----------------------------------------------------------------------------------------
# integer block sums and the product: fp64 brute force on dequantized blocks
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("t", [Q8_0, Q4_K, Q6_K, Q4_0, Q5_0])
def test_block_sums_equal_dequantized_dot(t):
    """'Products: weights against quantized activations': the integer block dot scaled by
    the float block scales equals the fp64 dot of the two dequantized blocks."""
    n_out, n_in, n_tok = 5, 512, 3
    W = oracle.quantize(t, synth.normal(31, (n_out, n_in), 0.5))
    X = synth.normal(32, (n_tok, n_in), 2.0)
    xt = oracle.VEC_DOT_TYPE[t]
    Xq = oracle.quantize(xt, X)
    S = oracle.block_sums(t, W, n_out, n_in, Xq, n_tok)
    wd = oracle.dequantize(t, W, n_in).astype(np.float64)
    xd = oracle.dequantize(xt, Xq, n_in).astype(np.float64)
    nb = n_in // oracle.BLOCK_ELEMS[t]
    be = oracle.BLOCK_ELEMS[t]
    wb, xb = oracle.BLOCK_BYTES[t], oracle.BLOCK_BYTES[xt]
    for tt in range(n_tok):
        for o in range(n_out):
            for k in range(nb):
                brute = float(np.dot(wd[o, k * be:(k + 1) * be], xd[tt, k * be:(k + 1) * be]))
                wblk = W[o, k * wb:(k + 1) * wb]
                xblk = Xq[tt, k * xb:(k + 1) * xb]
                if t in (Q8_0, Q4_0, Q5_0):
                    v = f16(int(wblk[0]) | int(wblk[1]) << 8) * f16(int(xblk[0]) | int(xblk[1]) << 8) * int(S[tt, o, k, 0])
                else:
                    dx = float(xblk[0:4].copy().view(np.float32)[0])
                    if t == Q4_K:
                        D = f16(int(wblk[0]) | int(wblk[1]) << 8)
                        Dm = f16(int(wblk[2]) | int(wblk[3]) << 8)
                        v = D * dx * int(S[tt, o, k, 0]) - Dm * dx * int(S[tt, o, k, 1])
                    else:
                        D = f16(int(wblk[208]) | int(wblk[209]) << 8)
                        v = D * dx * int(S[tt, o, k, 0])
                # the dequantized fp32 weights carry one rounding of S*q - M each (Q4_K)
                mag = float(np.dot(np.abs(wd[o, k * be:(k + 1) * be]), np.abs(xd[tt, k * be:(k + 1) * be])))
                assert abs(v - brute) <= 2 ** -23 * mag + 1e-300, (tt, o, k)


@pytest.mark.parametrize("t", [Q8_0, Q4_K, Q6_K, Q4_0, Q5_0])
def test_mul_mat_equals_fp64_brute_force(t):
    n_out, n_in, n_tok = 7, 768, 4
    W = oracle.quantize(t, synth.normal(41, (n_out, n_in), 0.02))
    X = synth.normal(42, (n_tok, n_in), 1.0)
    Y = oracle.mul_mat(t, W, n_out, n_in, X)
    xt = oracle.VEC_DOT_TYPE[t]
    wd = oracle.dequantize(t, W, n_in).astype(np.float64)
    xd = oracle.dequantize(xt, oracle.quantize(xt, X), n_in).astype(np.float64)
    ref = xd @ wd.T  # (n_tok, n_out): token-major, as ggml_mul_mat(W, X) = (X W^T)
    assert Y.shape == (n_tok, n_out)
    mag = np.abs(xd) @ np.abs(wd).T  # covers one fp32 rounding per dequantized weight
    assert np.all(np.abs(Y - ref) <= np.abs(ref) * 2 ** -23 + 2 ** -23 * mag)
    # activation rounding bound: |y_q - y_exact| <= sum_i |deq(w)_i| * d_x(block of i) / 2
    exact = X.astype(np.float64) @ wd.T
    be = oracle.BLOCK_ELEMS[xt]
    xq = oracle.quantize(xt, X).reshape(n_tok, n_in // be, -1)
    if xt == Q8_0:
        dx = np.array([[f16(int(b[0]) | int(b[1]) << 8) for b in row] for row in xq])
    else:
        dx = xq[:, :, 0:4].copy().view(np.float32)[:, :, 0].astype(np.float64)
    dx_el = np.repeat(dx, be, axis=1)
    bound = (dx_el / 2) @ np.abs(wd).T
    assert np.all(np.abs(Y - exact) <= bound * (1 + 1e-6) + 1e-6 * np.abs(exact))


@pytest.mark.parametrize("t", [Q8_0, Q4_K, Q6_K, Q4_0, Q5_0])
def test_mul_mat_orientation_example(t):
    """ggml_mul_mat(A, B^T) = C^T from the examples/simple page, with exact integers.

    The 2-wide operands are padded to one block: a pad column with 127 in the activation
    row (and 0 in the weights) makes the activation scale exactly 1; for Q8_0 a second
    pad column with 127 in the weights (and 0 in the activations) does the same for the
    weight scale.  For Q4_K/Q6_K the weight blocks are written field by field with scale 1.
    """
    g = read_fixture(os.path.join(GOLDEN, "mul_mat_orientation.txt"))
    A = np.array([[float(v) for v in r.split()] for r in g["A"].split(";")])
    BT = np.array([[float(v) for v in r.split()] for r in g["BT"].split(";")])
    CT = np.array([[float(v) for v in r.split()] for r in g["CT"].split(";")])
    n_in = oracle.BLOCK_ELEMS[t]
    X = np.zeros((3, n_in), np.float32)
    X[:, :2] = BT
    X[:, n_in - 1] = 127.0
    if t == Q8_0:
        Wf = np.zeros((4, n_in), np.float32)
        Wf[:, :2] = A
        Wf[:, n_in - 2] = 127.0
        W = oracle.quantize(Q8_0, Wf)
    elif t == Q4_K:
        W = np.zeros((4, 144), np.uint8)
        W[:, 0:2] = [0x00, 0x3C]          # d = 1
        W[:, 4:8] = 1                      # sc0..sc3 = 1, mins 0
        W[:, 12:16] = 0x01                 # sc4..sc7 = 1
        W[:, 16] = A[:, 0].astype(np.uint8)  # element 0 of sub-block 0 (low nibble)
        W[:, 17] = A[:, 1].astype(np.uint8)  # element 1
    elif t in (Q4_0, Q5_0):
        off = 8 if t == Q4_0 else 16
        W = np.zeros((4, oracle.BLOCK_BYTES[t]), np.uint8)
        W[:, 0:2] = [0x00, 0xBC]                       # d = -1: w = off - q covers 8 in Q4_0
        qs = 2 if t == Q4_0 else 6                     # first byte of the low-nibble codes
        codes = np.full((4, 32), off, np.int64)        # q = off: weight 0 elsewhere
        codes[:, :2] = off - A
        for i in range(32):
            l, hi = i % 16, i // 16
            W[:, qs + l] |= ((codes[:, i] & 15) << (4 * hi)).astype(np.uint8)
            if t == Q5_0:
                W[:, 2 + i // 8] |= (((codes[:, i] >> 4) & 1) << (i % 8)).astype(np.uint8)
    else:
        W = np.zeros((4, 210), np.uint8)
        W[:, 0] = A[:, 0].astype(np.uint8)   # low 4 bits of weight 0 (low nibble of ql[0])
        W[:, 1] = A[:, 1].astype(np.uint8)   # low 4 bits of weight 1 (low nibble of ql[1])
        W[:, 128:192] = 0xAA                 # top 2 bits = 2 for every weight: q - 32 = low bits
        W[:, 192:208] = 1                    # all sub-block scales 1
        W[:, 208:210] = [0x00, 0x3C]         # d = 1
    Y = oracle.mul_mat(t, W, 4, n_in, X)
    assert np.array_equal(Y, CT.astype(np.float32))


def test_mul_mat_sampled_and_threads_agree():
    t, n_out, n_in, n_tok = Q4_K, 37, 512, 5
    W = oracle.quantize(t, synth.normal(51, (n_out, n_in), 0.02))
    X = synth.normal(52, (n_tok, n_in))
    Y1 = oracle.mul_mat(t, W, n_out, n_in, X, n_threads=1)
    Y4 = oracle.mul_mat(t, W, n_out, n_in, X, n_threads=4)
    assert np.array_equal(Y1, Y4)
    rows, toks = np.array([0, 36, 5, 17]), np.array([4, 0, 2])
    Ys = oracle.mul_mat_sampled(t, W, n_out, n_in, X, rows, toks)
    assert np.array_equal(Ys, Y1[toks][:, rows])


# ----------------------------------------------------------------------------------------
# F16 weights: vec_dot_type F16 ("The GGML ecosystem, and where synapse fits", section 5:
# "F16 for F16"; "activations are rounded")
# ----------------------------------------------------------------------------------------

def test_f16_weights_are_ieee_half():
    """The F16 'format' is the IEEE binary16 value of each weight, little endian; checked
    against numpy's float16 cast (an independent RNE implementation)."""
    x = np.concatenate([_test_inputs(64).ravel(), np.array([65504.0, -65504.0, 6.0e-8, 2.0 ** -24], np.float32)])
    q = oracle.quantize(oracle.F16, x[None, :])
    assert np.array_equal(q.view("<u2")[0], x.astype(np.float16).view(np.uint16))
    back = oracle.dequantize(oracle.F16, q, x.size)[0]
    assert np.array_equal(back, x.astype(np.float16).astype(np.float32))
    # overflow to infinity and non-finite input are rejected
    assert oracle.quantize_status(oracle.F16, np.array([[7.0e4]], np.float32)) == -5
    assert oracle.quantize_status(oracle.F16, np.array([[np.inf]], np.float32)) == -5


def test_f16_mul_mat_is_the_half_product_in_fp64():
    """y = sum of fp16(w) * fp16(x) in exact arithmetic, rounded once to fp32."""
    n_out, n_in, n_tok = 6, 333, 4
    W = synth.normal(71, (n_out, n_in), 0.05)
    X = synth.normal(72, (n_tok, n_in), 3.0)
    Y = oracle.mul_mat(oracle.F16, oracle.quantize(oracle.F16, W), n_out, n_in, X)
    w16 = W.astype(np.float16).astype(np.float64)
    x16 = X.astype(np.float16).astype(np.float64)
    # each product is exact in fp64 (11-bit significands); the fp64 sum carries at most
    # n_in roundings of 2^-53 relative to the running magnitude
    ref = x16 @ w16.T
    mag = np.abs(x16) @ np.abs(w16).T
    assert np.all(np.abs(Y.astype(np.float64) - ref) <= 2 ** -24 * np.abs(ref) + n_in * 2 ** -52 * mag)
    with pytest.raises(oracle.OracleError):
        oracle.block_sums(oracle.F16, oracle.quantize(oracle.F16, W), n_out, n_in,
                          oracle.quantize(oracle.F16, X), n_tok)
