"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on the GPU.

Bar: quantized bytes, activation codes/scales/sums and integer block sums bit-exact;
fp32 products within |y - y_ref| <= 1e-4 * ||dequant(w_row)||_2 * ||x||_2 per element,
y_ref from the oracle (the same quantized-activation product in fp64).
"""
import numpy as np
import pytest

import oracle
from gguf_block_quantized_gb300 import synth, workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 1e-4
TYPES_W = [oracle.Q8_0, oracle.Q4_K, oracle.Q6_K, oracle.Q4_0, oracle.Q5_0]
TYPES_ALL = TYPES_W + [oracle.Q8_K]


@pytest.fixture(scope="module")
def syn():
    from gguf_block_quantized_gb300 import syn as s
    return s


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def tolerance(wtype, Wq, n_in, X):
    """Per-element bound 1e-4 * ||deq(w_row)|| * ||x|| as an (n_tok, n_out) array."""
    wd = oracle.dequantize(wtype, Wq, n_in).astype(np.float64)
    wn = np.sqrt((wd * wd).sum(axis=1))
    xn = np.sqrt((X.astype(np.float64) ** 2).sum(axis=1))
    return TOL * xn[:, None] * wn[None, :]


def assert_close(Y, ref, bound, what):
    err = np.abs(Y.astype(np.float64) - ref.astype(np.float64))
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"max err/bound {float((err / np.maximum(bound, 1e-300)).max()):.3g}")


def inputs_mixed(n_rows, n, seed):
    """Normal weights plus the degenerate rows the formats have."""
    x = synth.normal(seed, (n_rows, n), 0.02)
    if n_rows >= 8:
        x[1] = 0.0
        x[2] = synth.normal(seed + 1, n, 1e-6)          # fp16-subnormal scales
        x[3] = -np.abs(synth.normal(seed + 2, n, 1.0))  # all negative
        x[4] = np.abs(synth.normal(seed + 3, n, 1.0))   # all positive
        x[5] = 0.375                                      # constant
        x[6, ::7] *= 500.0                                # outliers
        x[7] = synth.uniform(seed + 4, n, -2.0, 2.0)
    return x


# ----------------------------------------------------------------------------------------
# quantize / dequantize: bit-exact
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("t", TYPES_ALL)
@pytest.mark.parametrize("shape", [(1, 256), (37, 512), (8, 4096), (300, 2304)])
def test_quantize_bit_exact(syn, t, shape):
    n_rows, n = shape
    x = inputs_mixed(n_rows, n, 100 + n_rows)
    want = oracle.quantize(t, x)
    got = host(syn.quantize(t, dev(x)))
    assert got.shape == want.shape
    mism = np.nonzero(got != want)
    assert mism[0].size == 0, f"{mism[0].size} bytes differ, first at {mism[0][:3]}, {mism[1][:3]}"


@pytest.mark.parametrize("t,name,n_sub", [(oracle.Q4_K, "q4_k_worked.txt", 8), (oracle.Q6_K, "q6_k_worked.txt", 16)])
def test_quantize_worked_blocks_bit_exact(syn, t, name, n_sub):
    """The hand-worked K-quant super-blocks (tests/golden; their scales, mins and codes are
    pinned on the CPU) encode to the same bytes on the GPU, alone and amid other rows."""
    import os
    from conftest import GOLDEN, read_fixture
    fx = read_fixture(os.path.join(GOLDEN, name))
    xb = np.concatenate([np.array([float(v) for v in fx[f"x{j}"].split()], np.float32) for j in range(n_sub)])
    x = inputs_mixed(9, 768, 55)
    x[0, :256] = xb
    x[4, 512:] = xb
    want = oracle.quantize(t, x)
    got = host(syn.quantize(t, dev(x)))
    assert np.array_equal(got, want)
    assert np.array_equal(got[0, :oracle.BLOCK_BYTES[t]], oracle.quantize(t, xb.reshape(1, 256))[0])


@pytest.mark.parametrize("t", TYPES_ALL)
def test_dequantize_bit_exact(syn, t):
    n_rows, n = 53, 1024
    q = oracle.quantize(t, inputs_mixed(n_rows, n, 7))
    want = oracle.dequantize(t, q, n)
    got = host(syn.dequantize(t, dev(q), n))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("t", [oracle.Q4_K, oracle.Q6_K])
def test_dequantize_f16_bit_exact(syn, t):
    """The fp16 expansion (the prefill's expanded weight operand): every value the oracle's
    fp32 dequantization rounded once to fp16, bit for bit, on quantized rows and on blocks of
    arbitrary bytes (every code, scale and sign pattern; non-finite halves left out)."""
    n_rows, n = 37, 2048
    Wq = oracle.quantize(t, synth.normal(1700 + t, (n_rows, n), 0.02))
    rng = np.random.default_rng(1710 + t)
    raw = rng.integers(0, 256, Wq.shape, dtype=np.uint8)
    bb = oracle.BLOCK_BYTES[t]
    blocks = raw.reshape(-1, bb)
    # keep the fp16 scales finite and small enough that no value overflows fp16
    d_off = (0,) if t == oracle.Q4_K else (208,)
    for o in d_off + ((2,) if t == oracle.Q4_K else ()):
        h = (rng.standard_normal(blocks.shape[0]) * 1e-3).astype(np.float16).view(np.uint8).reshape(-1, 2)
        blocks[:, o:o + 2] = h
    for W in (Wq, raw):
        ref = oracle.dequantize(t, W, n).astype(np.float32).astype(np.float16)
        got = host(syn.dequantize_f16(t, dev(W), n))
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("t", [oracle.Q4_K, oracle.Q6_K, oracle.Q8_0, oracle.Q4_0, oracle.Q5_0])
def test_dequantize_arbitrary_codes_bit_exact(syn, t):
    """Random block bytes (finite fp16 scales), including negative Q6_K scales."""
    n_rows, n = 19, 512
    rb = oracle.row_bytes(t, n)
    raw = synth.integers(3, (n_rows, rb), 0, 256).astype(np.uint8)
    nb, bb = n // oracle.BLOCK_ELEMS[t], oracle.BLOCK_BYTES[t]
    blocks = raw.reshape(n_rows, nb, bb)
    offs = {oracle.Q8_0: [0], oracle.Q4_K: [0, 2], oracle.Q6_K: [208], oracle.Q4_0: [0], oracle.Q5_0: [0]}[t]
    for o in offs:  # keep scales finite: clear the top exponent bit
        blocks[:, :, o + 1] &= 0xBF
    want = oracle.dequantize(t, raw, n)
    got = host(syn.dequantize(t, dev(raw), n))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_quantize_range_errors(syn):
    for t in TYPES_ALL:
        n = oracle.BLOCK_ELEMS[t]
        x = np.zeros((3, n), np.float32)
        x[2, 5] = np.nan
        with pytest.raises(syn.SynError) as e:
            syn.quantize(t, dev(x))
        assert e.value.status == syn.ERR_RANGE
    x = np.zeros((1, 256), np.float32)
    x[0, 0] = 1e9
    for t in (oracle.Q4_K, oracle.Q6_K, oracle.Q4_0, oracle.Q5_0):
        with pytest.raises(syn.SynError):
            syn.quantize(t, dev(x))
    syn.quantize(oracle.Q8_K, dev(x))  # fp32 scale: fine


# ----------------------------------------------------------------------------------------
# activation step and integer block sums: bit-exact
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("wt", TYPES_W)
def test_quantize_activations_bit_exact(syn, wt):
    n_tok, n_in = 5, 2048
    X = synth.activations(90, 0, n_tok, n_in)
    X[1] *= 1e-3
    X[2, :256] = 0.0
    xt = oracle.VEC_DOT_TYPE[wt]
    packed = oracle.quantize(xt, X)
    qs, d, bs = syn.quantize_activations(wt, dev(X))
    qs, d = host(qs), host(d)
    be, bb = oracle.BLOCK_ELEMS[xt], oracle.BLOCK_BYTES[xt]
    blocks = packed.reshape(n_tok, n_in // be, bb)
    if xt == oracle.Q8_0:
        want_d = oracle.fp16_bits_to_fp32(blocks[:, :, 0:2].copy().view(np.uint16)[:, :, 0])
        want_q = blocks[:, :, 2:].view(np.int8).reshape(n_tok, n_in)
    else:
        want_d = blocks[:, :, 0:4].copy().view(np.float32)[:, :, 0]
        want_q = blocks[:, :, 4:260].view(np.int8).reshape(n_tok, n_in)
        want_bs = blocks[:, :, 260:292].copy().view(np.int16).reshape(n_tok, n_in // 16)
        assert np.array_equal(host(bs), want_bs)
    assert np.array_equal(qs, want_q)
    assert np.array_equal(d.view(np.uint32), want_d.view(np.uint32))


def tie_rows(xt, n_in):
    """Activation rows whose quotients x / d sit exactly on, or within 2^-24 .. 2^-10 of, the
    half-integers where rounding turns (d exactly representable: amax = 127 * d)."""
    rng = np.random.default_rng(77)
    be = oracle.BLOCK_ELEMS[xt]
    rows = []
    for d in (1.0, 0.5, 3.0, 0.375, 2.0 ** -10, 6.103515625e-05):  # the last: fp16-subnormal edge
        x = np.empty(n_in, np.float64)
        for b0 in range(0, n_in, be):
            k = rng.integers(-126, 126, be).astype(np.float64)
            delta = rng.choice([0.0, 0.0, 2.0 ** -24, -2.0 ** -24, 2.0 ** -16, -2.0 ** -16, 2.0 ** -13, -2.0 ** -13,
                                2.0 ** -10], be)
            x[b0:b0 + be] = (k + 0.5 + delta) * d
            x[b0] = 127.0 * d  # the block maximum: d = amax / 127 exactly
        rows.append(x.astype(np.float32))
    return np.stack(rows)


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_K])
def test_quantize_activations_ties_bit_exact(syn, wt):
    """Values on and next to rounding ties of x / d: the encoders' multiply-by-reciprocal
    fast path must fall back to the division exactly where it could round differently."""
    xt = oracle.VEC_DOT_TYPE[wt]
    n_in = 1024
    X = tie_rows(xt, n_in)
    n_tok = X.shape[0]
    packed = oracle.quantize(xt, X)
    qs, d, bs = syn.quantize_activations(wt, dev(X))
    be, bb = oracle.BLOCK_ELEMS[xt], oracle.BLOCK_BYTES[xt]
    blocks = packed.reshape(n_tok, n_in // be, bb)
    off = 2 if xt == oracle.Q8_0 else 4
    want_q = blocks[:, :, off:off + be].view(np.int8).reshape(n_tok, n_in)
    assert np.array_equal(host(qs), want_q)
    # the same rows through syn_quantize (weights path of the same encoders)
    got = host(syn.quantize(xt, dev(X)))
    assert np.array_equal(got.reshape(-1), packed.reshape(-1))


@pytest.mark.parametrize("wt", TYPES_W)
def test_block_sums_bit_exact(syn, wt):
    n_out, n_in, n_tok = 9, 1024, 3
    W = oracle.quantize(wt, synth.normal(61, (n_out, n_in), 0.3))
    Xq = oracle.quantize(oracle.VEC_DOT_TYPE[wt], synth.normal(62, (n_tok, n_in)))
    want = oracle.block_sums(wt, W, n_out, n_in, Xq, n_tok)
    got = host(syn.block_sums(wt, dev(W), n_out, n_in, dev(Xq), n_tok))
    assert np.array_equal(got, want)


# ----------------------------------------------------------------------------------------
# mul_mat: decode kernel and tensor-core kernel against the oracle
# ----------------------------------------------------------------------------------------

def run_mul_mat(syn, wt, n_out, n_in, n_tok, seed, path, wstd=0.02):
    W32 = synth.normal(seed, (n_out, n_in), wstd)
    X = synth.normal(seed + 1, (n_tok, n_in))
    Wq = oracle.quantize(wt, W32)
    old = syn.set_gemv_max_tok(1 << 20 if path == "gemv" else 0)
    try:
        Y = host(syn.mul_mat(wt, dev(Wq), n_out, n_in, dev(X)))
    finally:
        syn.set_gemv_max_tok(old)
    assert syn.device_status() == syn.OK
    ref = oracle.mul_mat(wt, Wq, n_out, n_in, X, n_threads=8)
    return Y, ref, tolerance(wt, Wq, n_in, X)


# (77, 8192) and (40, 12288): rows of two stages' worth of blocks (split across warps, added into
# Y) and wider rows (several runs in one warp), per format
GEMV_SHAPES = [(1, 256, 1), (37, 512, 1), (300, 768, 2), (64, 2304, 3), (513, 1024, 4), (250, 4096, 8),
               (129, 512, 11), (77, 8192, 1), (40, 12288, 2)]


@pytest.mark.parametrize("wt", TYPES_W)
@pytest.mark.parametrize("shape", GEMV_SHAPES)
def test_mul_mat_gemv(syn, wt, shape):
    n_out, n_in, n_tok = shape
    Y, ref, bound = run_mul_mat(syn, wt, n_out, n_in, n_tok, 1000 + n_out, "gemv")
    assert_close(Y, ref, bound, f"gemv {shape}")


GEMM_SHAPES = [(128, 256, 16), (300, 1024, 40), (129, 512, 300), (1000, 2048, 256), (64, 4608, 33),
               (257, 768, 513)]


@pytest.mark.parametrize("wt", TYPES_W)
@pytest.mark.parametrize("shape", GEMM_SHAPES)
def test_mul_mat_gemm(syn, wt, shape):
    n_out, n_in, n_tok = shape
    Y, ref, bound = run_mul_mat(syn, wt, n_out, n_in, n_tok, 2000 + n_out, "gemm")
    assert_close(Y, ref, bound, f"gemm {shape}")


@pytest.mark.parametrize("wt", [oracle.Q4_K, oracle.Q6_K])
def test_mul_mat_gemm_tail_split(syn, wt):
    """160 row tiles on 152 SMs: whole tiles for the full wave, the last m-tiles split along K
    and added into their zeroed Y columns (ragged last tile), the other columns stored."""
    Y, ref, bound = run_mul_mat(syn, wt, 160 * 128 - 37, 1024, 16, 850 + wt, "gemm")
    assert_close(Y, ref, bound, "tail-split prefill")


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q5_0])
def test_mul_mat_row_not_multiple_of_256(syn, wt):
    # the 32-weight formats need only 32-element blocks: 800 = 25 blocks (ragged last k-step)
    for path in ("gemv", "gemm"):
        Y, ref, bound = run_mul_mat(syn, wt, 77, 800, 20, 77, path)
        assert_close(Y, ref, bound, f"{oracle.NAMES[wt]} n_in=800 {path}")


@pytest.mark.parametrize("n_tok", [1, 3, 8])
def test_mul_mat_batch_mixed_group(syn, n_tok):
    """Grouped decode of matrices of all three formats and ragged shapes in one call."""
    shapes = [(oracle.Q4_K, 300, 2048), (oracle.Q6_K, 77, 1024), (oracle.Q8_0, 129, 800),
              (oracle.Q4_K, 5, 256), (oracle.Q6_K, 1000, 512), (oracle.Q8_0, 64, 4096),
              (oracle.Q4_0, 200, 2048), (oracle.Q5_0, 99, 1024), (oracle.Q4_0, 17, 96)]
    items, refs = [], []
    for i, (wt, n_out, n_in) in enumerate(shapes):
        Wq = oracle.quantize(wt, synth.normal(300 + i, (n_out, n_in), 0.02))
        X = synth.normal(400 + i, (n_tok, n_in))
        Yd = torch.full((n_tok, n_out), float("nan"), device="cuda")
        items.append((wt, dev(Wq), n_out, n_in, dev(X), Yd))
        refs.append((oracle.mul_mat(wt, Wq, n_out, n_in, X), tolerance(wt, Wq, n_in, X)))
    syn.mul_mat_batch(items, n_tok)
    for (wt, _, n_out, n_in, _, Yd), (ref, bound) in zip(items, refs):
        assert_close(host(Yd), ref, bound, f"batch type {wt} {n_out}x{n_in}")
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("n_tok", [2, 3, 4])
def test_decode_rows_of_8_blocks(syn, n_tok):
    """Rows of 8 K-quant blocks (n_in = 2048, two rows per warp step) at 2-4 tokens: single
    products with an odd row count (a last warp step of one row), a narrow product
    (activations converted in the decode CTAs), and a grouped call mixing them with 4096-wide
    rows and Q8_0."""
    cases = [[(oracle.Q4_K, 1001, 2048)], [(oracle.Q6_K, 2047, 2048)], [(oracle.Q6_K, 37, 2048)],
             [(oracle.Q4_K, 512, 2048), (oracle.Q6_K, 301, 2048), (oracle.Q4_K, 129, 4096),
              (oracle.Q8_0, 200, 2048), (oracle.Q6_K, 64, 2048)]]
    for c, shapes in enumerate(cases):
        items, refs = [], []
        for i, (wt, n_out, n_in) in enumerate(shapes):
            Wq = oracle.quantize(wt, synth.normal(1500 + 10 * c + i, (n_out, n_in), 0.02))
            X = synth.normal(1600 + 10 * c + i, (n_tok, n_in))
            Yd = torch.full((n_tok, n_out), float("nan"), device="cuda")
            items.append((wt, dev(Wq), n_out, n_in, dev(X), Yd))
            refs.append((oracle.mul_mat(wt, Wq, n_out, n_in, X), tolerance(wt, Wq, n_in, X)))
        syn.mul_mat_batch(items, n_tok)
        for (wt, _, n_out, n_in, _, Yd), (ref, bound) in zip(items, refs):
            assert_close(host(Yd), ref, bound, f"rows of 8 blocks {oracle.NAMES[wt]} {n_out}x{n_in} n_tok {n_tok}")
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("n_tok", [1, 3, 6, 300])
def test_mul_mat_batch_shared_inputs(syn, n_tok):
    """A grouped call whose products share activation inputs (q/k/v on one input, gate/up on
    another, formats with the same activation layout or not): each shared input is converted
    once per layout, on the decode path (one conversion unit feeds several products, and one
    shared-memory copy serves the CTA's products) and on the prefill path; every product
    matches the oracle, and matches its own syn_mul_mat."""
    n_in = 1024
    XA, XF = synth.normal(610, (n_tok, n_in)), synth.normal(611, (n_tok, n_in))
    specs = [(oracle.Q4_K, 384, XA), (oracle.Q4_K, 128, XA), (oracle.Q6_K, 128, XA), (oracle.Q8_0, 256, XA),
             (oracle.F16, 64, XA), (oracle.Q4_K, 640, XF), (oracle.Q4_K, 640, XF), (oracle.Q5_0, 96, XF),
             (oracle.Q4_0, 64, XF), (oracle.Q8_0, 32, XA)]
    XAd, XFd = dev(XA), dev(XF)
    items, refs, singles = [], [], []
    for i, (wt, n_out, X) in enumerate(specs):
        Wq = oracle.quantize(wt, synth.normal(620 + i, (n_out, n_in), 0.02))
        Wd = dev(Wq)
        Xd = XAd if X is XA else XFd
        items.append((wt, Wd, n_out, n_in, Xd, torch.full((n_tok, n_out), np.nan, device="cuda")))
        refs.append((oracle.mul_mat(wt, Wq, n_out, n_in, X), tolerance(wt, Wq, n_in, X)))
        singles.append(host(syn.mul_mat(wt, Wd, n_out, n_in, Xd)))
    syn.mul_mat_batch(items, n_tok)
    for (wt, _, n_out, _, _, Yd), (ref, bound), y1 in zip(items, refs, singles):
        y = host(Yd)
        assert_close(y, ref, bound, f"shared-input batch type {wt} {n_out}x{n_in} n_tok {n_tok}")
        assert_close(y, y1, 2 * bound, f"batch vs single type {wt} {n_out}")
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("wt,n_out,n_in,n_tok", [
    (oracle.Q4_K, 333, 8192, 70), (oracle.Q6_K, 130, 14336, 33), (oracle.Q8_0, 258, 8192, 20),
    (oracle.Q4_0, 256, 8192, 48), (oracle.Q5_0, 129, 8192, 17), (oracle.F16, 96, 8192, 50),
    (oracle.Q4_K, 640, 14336, 300)])
def test_streamk_prefill(syn, wt, n_out, n_in, n_tok):
    """Products whose tiles do not fill one wave and whose K is long (>= 32 super-steps) run
    on the stream-K schedule: every CTA an equal range of tile x K work, partial tiles added
    into a zeroed Y (by TMA reduce-adds, or element-wise where the Y pitch is not a multiple of
    16 bytes).  Ragged rows and tokens; every format; against the oracle."""
    Y, ref, bound = run_mul_mat(syn, wt, n_out, n_in, n_tok, 1300 + n_out, "gemm")
    assert_close(Y, ref, bound, f"stream-K {oracle.NAMES[wt]} {n_out}x{n_in} n_tok {n_tok}")
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("wt,n_out,n_in,n_tok", [(oracle.Q4_K, 1400, 8192, 40), (oracle.Q6_K, 876, 8192, 300)])
def test_streamk_tail_prefill(syn, wt, n_out, n_in, n_tok):
    """Products with more tiles than SMs and long K (here on 8 SMs: 11 tiles of one token
    tile, and 14 tiles of two) run whole tiles for the full waves, then share the tiles of the
    last wave stream-K (their Y columns zeroed, partial tiles added); against the oracle."""
    prev = syn.set_sm_limit(8)
    try:
        Y, ref, bound = run_mul_mat(syn, wt, n_out, n_in, n_tok, 1350 + n_out, "gemm")
    finally:
        syn.set_sm_limit(prev)
    assert_close(Y, ref, bound, f"stream-K tail {oracle.NAMES[wt]} {n_out}x{n_in} n_tok {n_tok}")
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("wt,n_out,n_in,n_tok", [(oracle.Q4_K, 300, 1024, 40), (oracle.Q6_K, 131, 768, 60),
                                                 (oracle.Q4_K, 257, 4096, 300), (oracle.Q6_K, 129, 512, 1600)])
def test_prefill_expanded_weights(syn, wt, n_out, n_in, n_tok):
    """Prefill with the K-quant weights expanded to fp16 first (forced at every token count
    here; by default from 1536 tokens), then the fp16 tensor-core product; the last case runs
    at the default threshold.  Ragged rows and token tiles; against the oracle."""
    prev = syn.set_prefill_expand_tok(0 if n_tok < 1536 else -1)
    try:
        Y, ref, bound = run_mul_mat(syn, wt, n_out, n_in, n_tok, 1400 + n_out, "gemm")
    finally:
        syn.set_prefill_expand_tok(prev)
    assert_close(Y, ref, bound, f"expanded {oracle.NAMES[wt]} {n_out}x{n_in} n_tok {n_tok}")
    assert syn.device_status() == syn.OK


def test_prefill_expanded_weights_grouped(syn):
    """A grouped prefill call with expanded weights: q/k/v-like products on one input (one
    conversion, the fp16 weight buffer reused product by product), a Q8_0 product (not
    expanded) in the same group, and a split-tail product (on 8 SMs); against the oracle."""
    n_tok, n_in = 96, 2048
    shapes = [(oracle.Q4_K, 512), (oracle.Q6_K, 129), (oracle.Q8_0, 200), (oracle.Q4_K, 1100)]
    X = synth.normal(1450, (n_tok, n_in))
    Xd = dev(X)
    items, refs = [], []
    for i, (wt, n_out) in enumerate(shapes):
        Wq = oracle.quantize(wt, synth.normal(1460 + i, (n_out, n_in), 0.02))
        Yd = torch.full((n_tok, n_out), float("nan"), device="cuda")
        items.append((wt, dev(Wq), n_out, n_in, Xd, Yd))
        refs.append((oracle.mul_mat(wt, Wq, n_out, n_in, X), tolerance(wt, Wq, n_in, X)))
    prev, lim = syn.set_prefill_expand_tok(0), syn.set_sm_limit(8)
    try:
        syn.mul_mat_batch(items, n_tok)
    finally:
        syn.set_prefill_expand_tok(prev)
        syn.set_sm_limit(lim)
    for (wt, _, n_out, _, _, Yd), (ref, bound) in zip(items, refs):
        assert_close(host(Yd), ref, bound, f"expanded group {oracle.NAMES[wt]} {n_out}")
    assert syn.device_status() == syn.OK


def test_prepared_batch_matches_grouped_call(syn):
    """The prepared grouped call (descriptors marshalled once) runs the same launches as
    mul_mat_batch: bit-identical outputs, and repeated calls see updated inputs."""
    shapes = [(oracle.Q4_K, 512, 2048), (oracle.Q6_K, 256, 2048), (oracle.Q8_0, 300, 1024)]
    Ws = [dev(oracle.quantize(wt, synth.normal(70 + k, (n_out, n_in), 0.02))) for k, (wt, n_out, n_in) in enumerate(shapes)]
    for n_tok in (1, 3):
        Xs = [dev(synth.normal(80 + k, (n_tok, n_in))) for k, (_, _, n_in) in enumerate(shapes)]
        Ya = [torch.full((n_tok, n_out), np.nan, device="cuda") for _, n_out, _ in shapes]
        Yb = [torch.full((n_tok, n_out), np.nan, device="cuda") for _, n_out, _ in shapes]
        syn.mul_mat_batch([(wt, W, n_out, n_in, X, Y) for (wt, n_out, n_in), W, X, Y in zip(shapes, Ws, Xs, Ya)], n_tok)
        pb = syn.prepare_batch([(wt, W, n_out, n_in, X, Y) for (wt, n_out, n_in), W, X, Y in zip(shapes, Ws, Xs, Yb)],
                               n_tok, stream=torch.cuda.current_stream())
        pb()
        for a, b in zip(Ya, Yb):
            assert torch.equal(a, b)
        for X in Xs:
            X.mul_(-1.0)  # the next call reads the new contents of the same buffers
        pb()
        for a, b in zip(Ya, Yb):
            assert torch.equal(-a, b)
    assert syn.device_status() == syn.OK


def test_staged_batch_host_buffers(syn):
    """The host-staged grouped call (inputs copied in from pinned host memory, outputs copied
    out) gives the device path's outputs, bit for bit, in the host buffer."""
    shapes = [(oracle.Q4_K, 512, 2048), (oracle.Q6_K, 256, 2048), (oracle.Q4_0, 96, 512)]
    n_tok = 2
    xo, yo = [0], [0]
    for _, n_out, n_in in shapes:
        xo.append(xo[-1] + n_tok * n_in)
        yo.append(yo[-1] + n_tok * n_out)
    xh = torch.from_numpy(synth.normal(700, (xo[-1],))).pin_memory()
    yh = torch.full((yo[-1],), np.nan).pin_memory()
    xd, yd = torch.empty(xo[-1], device="cuda"), torch.empty(yo[-1], device="cuda")
    Ws = [dev(oracle.quantize(wt, synth.normal(710 + k, (n_out, n_in), 0.02))) for k, (wt, n_out, n_in) in enumerate(shapes)]
    items = [(wt, Ws[k], n_out, n_in, xd[xo[k]:xo[k + 1]].view(n_tok, n_in), yd[yo[k]:yo[k + 1]].view(n_tok, n_out))
             for k, (wt, n_out, n_in) in enumerate(shapes)]
    stream = torch.cuda.current_stream()
    pb = syn.prepare_batch(items, n_tok, stream=stream, staged=(xh, xd, yd, yh))
    pb()
    stream.synchronize()
    got = yh.numpy().copy()
    assert np.array_equal(xd.cpu().numpy(), xh.numpy())
    yd.fill_(float("nan"))
    syn.mul_mat_batch(items, n_tok, stream=stream)  # the same launches on the staged inputs
    assert np.array_equal(got, host(yd))
    X = xh.numpy()
    for k, (wt, n_out, n_in) in enumerate(shapes):
        Wq = oracle.quantize(wt, synth.normal(710 + k, (n_out, n_in), 0.02))
        Xk = X[xo[k]:xo[k + 1]].reshape(n_tok, n_in)
        assert_close(got[yo[k]:yo[k + 1]].reshape(n_tok, n_out), oracle.mul_mat(wt, Wq, n_out, n_in, Xk),
                     tolerance(wt, Wq, n_in, Xk), f"staged type {wt}")
    assert syn.device_status() == syn.OK


def test_decode_plans_interleaved(syn):
    """Grouped decode calls of different shapes interleaved (the host keeps the last few work
    partitions by shape): every call matches the oracle, and repeats are bit-identical."""
    cfgs = [([(oracle.Q4_K, 2048, 2048), (oracle.Q6_K, 512, 2048)], 1),
            ([(oracle.Q8_0, 4096, 1024), (oracle.Q4_0, 300, 512), (oracle.Q5_0, 777, 1024)], 2),
            ([(oracle.Q4_K, 8192, 2048)], 1),
            ([(oracle.Q6_K, 2048, 8192), (oracle.Q4_K, 512, 2048)], 3),
            ([(oracle.Q4_K, 8192, 2048)], 5),
            ([(oracle.Q8_0, 64, 256)], 1)]
    data = []
    for c, (shapes, n_tok) in enumerate(cfgs):
        Wq = [oracle.quantize(wt, synth.normal(90 + 7 * c + k, (n_out, n_in), 0.02)) for k, (wt, n_out, n_in) in enumerate(shapes)]
        Xs = [synth.normal(95 + 7 * c + k, (n_tok, n_in)) for k, (_, _, n_in) in enumerate(shapes)]
        data.append((shapes, n_tok, [dev(w) for w in Wq], [dev(x) for x in Xs], Wq, Xs))
    old = syn.set_gemv_max_tok(8)
    try:
        first = {}
        for rnd in range(3):
            for c, (shapes, n_tok, Wd, Xd, Wq, Xs) in enumerate(data):
                Ys = [torch.full((n_tok, n_out), np.nan, device="cuda") for _, n_out, _ in shapes]
                syn.mul_mat_batch([(wt, W, n_out, n_in, X, Y) for (wt, n_out, n_in), W, X, Y in zip(shapes, Wd, Xd, Ys)], n_tok)
                got = [host(Y) for Y in Ys]
                if rnd == 0:
                    for (wt, n_out, n_in), w, x, y in zip(shapes, Wq, Xs, got):
                        ref = oracle.mul_mat(wt, w, n_out, n_in, x)
                        assert_close(y, ref, tolerance(wt, w, n_in, x), f"cfg {c} type {wt} {n_out}x{n_in}")
                    first[c] = got
                else:
                    for a, b in zip(first[c], got):
                        assert np.array_equal(a, b), f"cfg {c} round {rnd}"
    finally:
        syn.set_gemv_max_tok(old)
    assert syn.device_status() == syn.OK


def test_mul_mat_orientation_example_exact(syn):
    """ggml_mul_mat(A, B^T) = C^T with the examples/simple integers, exact on both paths."""
    A = np.array([[2, 8], [5, 1], [4, 2], [8, 6]], np.float32)
    BT = np.array([[10, 5], [9, 9], [5, 4]], np.float32)
    CT = np.array([[60, 55, 50, 110], [90, 54, 54, 126], [42, 29, 28, 64]], np.float32)
    W = np.zeros((4, 32), np.float32); W[:, :2] = A; W[:, 30] = 127.0
    X = np.zeros((3, 32), np.float32); X[:, :2] = BT; X[:, 31] = 127.0
    Wq = oracle.quantize(oracle.Q8_0, W)
    for n in (1 << 20, 0):
        old = syn.set_gemv_max_tok(n)
        try:
            Y = host(syn.mul_mat(oracle.Q8_0, dev(Wq), 4, 32, dev(X)))
        finally:
            syn.set_gemv_max_tok(old)
        assert np.array_equal(Y, CT)


def test_gemv_and_gemm_agree(syn):
    wt, n_out, n_in, n_tok = oracle.Q4_K, 384, 2048, 8
    W = oracle.quantize(wt, synth.normal(5, (n_out, n_in), 0.02))
    X = synth.normal(6, (n_tok, n_in))
    outs = []
    for n in (1 << 20, 0):
        old = syn.set_gemv_max_tok(n)
        try:
            outs.append(host(syn.mul_mat(wt, dev(W), n_out, n_in, dev(X))))
        finally:
            syn.set_gemv_max_tok(old)
    assert_close(outs[0], outs[1], 2 * tolerance(wt, W, n_in, X), "gemv vs gemm")


def test_gemv_deterministic(syn):
    wt, n_out, n_in = oracle.Q6_K, 1000, 4096
    W = dev(oracle.quantize(wt, synth.normal(8, (n_out, n_in), 0.02)))
    X = dev(synth.normal(9, (2, n_in)))
    a = host(syn.mul_mat(wt, W, n_out, n_in, X))
    b = host(syn.mul_mat(wt, W, n_out, n_in, X))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_gemv_split_rows_deterministic(syn):
    """Rows whose two runs go to different warps are added into Y: the result must not depend
    on the order of the two additions (bit-identical across calls) and must match the oracle."""
    shapes = [(oracle.Q6_K, 600, 8192), (oracle.Q4_K, 200, 12288), (oracle.Q8_0, 333, 8192)]
    items, refs = [], []
    for i, (wt, n_out, n_in) in enumerate(shapes):
        Wq = oracle.quantize(wt, synth.normal(500 + i, (n_out, n_in), 0.02))
        X = synth.normal(600 + i, (2, n_in))
        items.append((wt, dev(Wq), n_out, n_in, dev(X), torch.full((2, n_out), float("nan"), device="cuda")))
        refs.append((oracle.mul_mat(wt, Wq, n_out, n_in, X), tolerance(wt, Wq, n_in, X)))
    outs = []
    for _ in range(3):
        syn.mul_mat_batch(items, 2)
        outs.append([host(it[5]).copy() for it in items])
    for k in range(len(shapes)):
        assert_close(outs[0][k], refs[k][0], refs[k][1], f"split rows {shapes[k]}")
        for o in outs[1:]:
            assert np.array_equal(o[k].view(np.uint32), outs[0][k].view(np.uint32))
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("n_tok", [1, 3])
def test_decode_chain_back_to_back(syn, n_tok):
    """Dependent decode steps enqueued back to back: step i+1 reads step i's output as its
    input, every step reuses the library's workspace, and a split-row product adds into the
    same Y every step.  The conversion launch of step i+1 starts while step i's decode launch
    drains (programmatic dependent launch) and must wait for it: the results, eager and
    replayed from one CUDA graph, are bit-identical to the same calls with a device
    synchronisation between them, and the first step matches the oracle."""
    L, d = 5, 2048
    Wa = [oracle.quantize(oracle.Q4_K, synth.normal(700 + i, (d, d), 0.02)) for i in range(L)]
    Wb = [oracle.quantize(oracle.Q6_K, synth.normal(720 + i, (1024, d), 0.02)) for i in range(L)]
    Ws = oracle.quantize(oracle.Q6_K, synth.normal(740, (600, 8192), 0.02))  # rows split in two runs
    Wa_d, Wb_d, Ws_d = [dev(w) for w in Wa], [dev(w) for w in Wb], dev(Ws)
    X0 = synth.normal(741, (n_tok, d))
    X0_d = dev(X0)
    X8 = dev(synth.normal(742, (n_tok, 8192)))
    stream = torch.cuda.Stream()

    def buffers():
        nan = float("nan")
        return ([torch.full((n_tok, d), nan, device="cuda") for _ in range(L)],
                [torch.full((n_tok, 1024), nan, device="cuda") for _ in range(L)],
                torch.full((n_tok, 600), nan, device="cuda"))

    def run(bufs, sync):
        Ya, Yb, Ys = bufs
        x = X0_d
        for i in range(L):
            syn.mul_mat_batch([(oracle.Q4_K, Wa_d[i], d, d, x, Ya[i]), (oracle.Q6_K, Wb_d[i], 1024, d, x, Yb[i]),
                               (oracle.Q6_K, Ws_d, 600, 8192, X8, Ys)], n_tok, stream=stream)
            if sync:
                torch.cuda.synchronize()
            x = Ya[i]

    def fetch(bufs):
        torch.cuda.synchronize()
        Ya, Yb, Ys = bufs
        return [host(y).copy() for y in Ya + Yb + [Ys]]

    with torch.cuda.stream(stream):
        ref_bufs = buffers()
        run(ref_bufs, True)
        ref = fetch(ref_bufs)
        eager = buffers()
        run(eager, False)
        got = [fetch(eager)]
    graph_bufs = buffers()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run(graph_bufs, False)
    for _ in range(2):
        for y in graph_bufs[0] + graph_bufs[1] + [graph_bufs[2]]:
            y.fill_(float("nan"))
        g.replay()
        got.append(fetch(graph_bufs))
    for out in got:
        for k, (a, b) in enumerate(zip(out, ref)):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"output {k} differs"
    assert_close(ref[0], oracle.mul_mat(oracle.Q4_K, Wa[0], d, d, X0), tolerance(oracle.Q4_K, Wa[0], d, X0), "step 0")
    X8h = host(X8)
    assert_close(ref[-1], oracle.mul_mat(oracle.Q6_K, Ws, 600, 8192, X8h), tolerance(oracle.Q6_K, Ws, 8192, X8h),
                 "split rows")
    assert syn.device_status() == syn.OK


DET_SHAPES = [(300, 1024, 37), (600, 8192, 11), (77, 2304, 9)]  # (n_out, n_in, n_tok); 8192: rows split by default


@pytest.mark.parametrize("wt", TYPES_W + [oracle.F16])
@pytest.mark.parametrize("shape", DET_SHAPES)
def test_deterministic_mode_invariants(syn, wt, shape):
    """Deterministic mode (G1, D1 of synapse): a token's output row is bit-identical whatever
    the other tokens of the call (prefill rows equal decode rows), whatever the SM limit,
    the grouping of products into one batch call or the split of the tokens into calls;
    and it is within the product's tolerance of the oracle."""
    n_out, n_in, n_tok = shape
    Wq = oracle.quantize(wt, synth.normal(800 + n_in, (n_out, n_in), 0.02))
    X = synth.normal(801 + n_in, (n_tok, n_in))
    W, Xd = dev(Wq), dev(X)
    old = syn.set_deterministic(True)
    try:
        ref = host(syn.mul_mat(wt, W, n_out, n_in, Xd))
        outs = {"one token per call": np.concatenate([host(syn.mul_mat(wt, W, n_out, n_in, Xd[t:t + 1]))
                                                      for t in range(n_tok)]),
                "calls of 5 tokens": np.concatenate([host(syn.mul_mat(wt, W, n_out, n_in, Xd[t:t + 5]))
                                                     for t in range(0, n_tok, 5)])}
        for lim in (1, 13, 100):
            prev = syn.set_sm_limit(lim)
            try:
                outs[f"{lim} SMs"] = host(syn.mul_mat(wt, W, n_out, n_in, Xd))
            finally:
                syn.set_sm_limit(prev)
        # grouped with two other products in one batch call (decode-sized token count)
        if wt != oracle.F16:
            Wo = dev(oracle.quantize(oracle.Q6_K, synth.normal(802, (129, 8192), 0.02)))
            Xo = dev(synth.normal(803, (n_tok, 8192)))
            Yb = torch.full((n_tok, n_out), float("nan"), device="cuda")
            Yb2 = torch.full((n_tok, n_out), float("nan"), device="cuda")
            Yo = [torch.empty((n_tok, 129), device="cuda") for _ in range(2)]
            syn.mul_mat_batch([(oracle.Q6_K, Wo, 129, 8192, Xo, Yo[0]), (wt, W, n_out, n_in, Xd, Yb),
                               (oracle.Q6_K, Wo, 129, 8192, Xo, Yo[1]), (wt, W, n_out, n_in, Xd, Yb2)], n_tok)
            outs["batched"] = host(Yb)
            outs["batched, input shared with another product"] = host(Yb2)
        for what, Y in outs.items():
            assert np.array_equal(Y.view(np.uint32), ref.view(np.uint32)), what
    finally:
        syn.set_deterministic(old)
    assert_close(ref, oracle.mul_mat(wt, Wq, n_out, n_in, X), tolerance(wt, Wq, n_in, X), "deterministic vs oracle")
    assert syn.device_status() == syn.OK


def test_deterministic_mode_rejects_too_wide_rows(syn):
    """A row whose converted activations do not fit the decode kernel's shared memory is
    rejected in deterministic mode (the tensor-core prefill takes it otherwise)."""
    wt, n_out, n_in = oracle.Q4_K, 3, 98304
    Wq = oracle.quantize(wt, synth.normal(810, (n_out, n_in), 0.02))
    X = synth.normal(811, (1, n_in))
    W, Xd = dev(Wq), dev(X)
    Y = torch.empty((1, n_out), device="cuda")
    old = syn.set_deterministic(True)
    try:
        assert syn.syn_mul_mat(wt, syn._ptr(W), n_out, n_in, syn._ptr(Xd), 1, syn._ptr(Y), None) == syn.ERR_SHAPE
    finally:
        syn.set_deterministic(old)
    Y = host(syn.mul_mat(wt, W, n_out, n_in, Xd))
    assert_close(Y, oracle.mul_mat(wt, Wq, n_out, n_in, X), tolerance(wt, Wq, n_in, X), "wide row, default mode")


# the widest rows the decode kernel takes (converted activations of one token within its
# shared-memory budget), as documented with syn_set_deterministic
DECODE_MAX_N_IN = {oracle.Q4_K: 72960, oracle.Q6_K: 72960, oracle.Q8_0: 74112, oracle.Q4_0: 70208, oracle.Q5_0: 70208}


@pytest.mark.parametrize("wt", sorted(DECODE_MAX_N_IN))
def test_decode_widest_rows(syn, wt):
    """At the documented widest row the decode kernels run it (deterministic mode accepts it)
    and match the oracle; one block wider is rejected in that mode."""
    n_out, n_in = 5, DECODE_MAX_N_IN[wt]
    be = 256 if wt in (oracle.Q4_K, oracle.Q6_K) else 32
    Wq = oracle.quantize(wt, synth.normal(820 + wt, (n_out, n_in + be), 0.02))
    X = synth.normal(830 + wt, (2, n_in + be))
    old = syn.set_deterministic(True)
    try:
        Wn = oracle.quantize(wt, synth.normal(820 + wt, (n_out, n_in), 0.02))
        Xn = np.ascontiguousarray(X[:, :n_in])
        Y = host(syn.mul_mat(wt, dev(Wn), n_out, n_in, dev(Xn)))
        W2, X2 = dev(Wq), dev(X)
        Y2 = torch.empty((2, n_out), device="cuda")
        assert syn.syn_mul_mat(wt, syn._ptr(W2), n_out, n_in + be, syn._ptr(X2), 2, syn._ptr(Y2), None) == syn.ERR_SHAPE
    finally:
        syn.set_deterministic(old)
    assert_close(Y, oracle.mul_mat(wt, Wn, n_out, n_in, Xn), tolerance(wt, Wn, n_in, Xn), f"widest row {n_in}")
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("wt", [oracle.Q4_K, oracle.Q8_0])
def test_mul_mat_gemm_many_token_tiles(syn, wt):
    """Prefill over 17 token tiles of 256 with a ragged last one, and a ragged row count."""
    Y, ref, bound = run_mul_mat(syn, wt, 130, 512, 4097, 840 + wt, "gemm")
    assert_close(Y, ref, bound, "4097 tokens")


@pytest.mark.parametrize("lim", [1, 7, 64])
def test_sm_limit_parity(syn, lim):
    """Products on a limited number of SMs (decode, grouped decode and tensor-core prefill)
    stay within tolerance of the oracle."""
    prev = syn.set_sm_limit(lim)
    try:
        for wt, n_out, n_in, n_tok in [(oracle.Q4_K, 300, 2048, 1), (oracle.Q6_K, 129, 8192, 3),
                                      (oracle.Q8_0, 257, 1024, 40), (oracle.Q4_K, 200, 768, 130)]:
            Y, ref, bound = run_mul_mat(syn, wt, n_out, n_in, n_tok, 820 + lim, "gemv" if n_tok <= 8 else "gemm")
            assert_close(Y, ref, bound, f"{oracle.NAMES[wt]} {n_out}x{n_in} tok={n_tok} on {lim} SMs")
    finally:
        syn.set_sm_limit(prev)
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("wt", [oracle.Q4_K, oracle.Q6_K, oracle.Q8_0, oracle.Q4_0, oracle.Q5_0, oracle.F16])
def test_default_per_format_threshold(syn, wt):
    """The default (per-format) decode/prefill choice: token counts on both sides of each
    format's crossover, single and grouped, against the oracle."""
    n_out, n_in = 136, 768
    Wq = oracle.quantize(wt, synth.normal(40 + wt, (n_out, n_in), 0.02))
    old = syn.set_gemv_max_tok(-1)
    try:
        for n_tok in (1, 2, 3, 4, 5, 8, 9):
            X = synth.normal(50 + n_tok, (n_tok, n_in))
            ref = oracle.mul_mat(wt, Wq, n_out, n_in, X)
            bound = tolerance(wt, Wq, n_in, X)
            assert_close(host(syn.mul_mat(wt, dev(Wq), n_out, n_in, dev(X))), ref, bound, f"type {wt} n_tok {n_tok}")
            Wd, Xd = dev(Wq), dev(X)
            Y1, Y2 = (torch.full((n_tok, n_out), np.nan, device="cuda") for _ in range(2))
            syn.mul_mat_batch([(wt, Wd, n_out, n_in, Xd, Y1), (oracle.Q4_K, Wd if wt == oracle.Q4_K else
                               dev(oracle.quantize(oracle.Q4_K, synth.normal(60, (n_out, n_in), 0.02))),
                               n_out, n_in, Xd, Y2)], n_tok)
            assert_close(host(Y1), ref, bound, f"batch type {wt} n_tok {n_tok}")
            assert np.isfinite(host(Y2)).all()
    finally:
        assert syn.set_gemv_max_tok(old) == -1
    assert syn.device_status() == syn.OK


def test_mul_mat_zero_and_degenerate(syn):
    wt, n_out, n_in = oracle.Q4_K, 40, 512
    Wq = oracle.quantize(wt, inputs_mixed(n_out, n_in, 3))
    X = synth.normal(4, (5, n_in))
    X[2] = 0.0
    for n in (1 << 20, 0):
        old = syn.set_gemv_max_tok(n)
        try:
            Y = host(syn.mul_mat(wt, dev(Wq), n_out, n_in, dev(X)))
        finally:
            syn.set_gemv_max_tok(old)
        ref = oracle.mul_mat(wt, Wq, n_out, n_in, X)
        assert_close(Y, ref, tolerance(wt, Wq, n_in, X), "degenerate rows")
        assert np.all(Y[2] == 0.0) and np.all(Y[:, 1] == 0.0)
    # n_tok == 0 is a no-op
    Y = torch.full((0, n_out), 1.0, device="cuda")
    syn.mul_mat(wt, dev(Wq), n_out, n_in, torch.zeros((0, n_in), device="cuda"), Y=Y)


def test_mul_mat_error_codes(syn):
    Wq = dev(oracle.quantize(oracle.Q4_K, synth.normal(1, (4, 256), 0.02)))
    X = torch.zeros((1, 256), device="cuda")
    Y = torch.zeros((1, 4), device="cuda")
    s = 0
    assert syn.syn_mul_mat(oracle.Q8_K, Wq.data_ptr(), 4, 256, X.data_ptr(), 1, Y.data_ptr(), s) == syn.ERR_TYPE
    assert syn.syn_mul_mat(oracle.Q4_K, Wq.data_ptr(), 4, 100, X.data_ptr(), 1, Y.data_ptr(), s) == syn.ERR_SHAPE
    assert syn.syn_mul_mat(oracle.Q4_K, None, 4, 256, X.data_ptr(), 1, Y.data_ptr(), s) == syn.ERR_NULL
    assert syn.syn_mul_mat(oracle.Q4_K, Wq.data_ptr() + 2, 4, 256, X.data_ptr(), 1, Y.data_ptr(), s) == syn.ERR_ALIGN


# ----------------------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times: sampled entries
# ----------------------------------------------------------------------------------------

def sampled_check(syn, m, n_tok, workload, index, n_rows=48, n_toks=4, path=None):
    W32 = synth.weight(workload, index, m.n_out, m.n_in)
    X = synth.activations(workload, index, n_tok, m.n_in)
    Wq = oracle.quantize(m.wtype, W32)
    old = syn.set_gemv_max_tok(-1 if path is None else (1 << 20 if path == "gemv" else 0))
    try:
        Y = host(syn.mul_mat(m.wtype, dev(Wq), m.n_out, m.n_in, dev(X)))
    finally:
        syn.set_gemv_max_tok(old)
    rows = np.unique(np.concatenate([[0, m.n_out - 1], synth.integers(index, n_rows, 0, m.n_out)]))
    toks = np.unique(np.concatenate([[0, n_tok - 1], synth.integers(index + 1, n_toks, 0, n_tok)]))
    ref = oracle.mul_mat_sampled(m.wtype, Wq, m.n_out, m.n_in, X, rows, toks)
    wd = oracle.dequantize(m.wtype, Wq[rows], m.n_in).astype(np.float64)
    bound = TOL * np.sqrt((X[toks].astype(np.float64) ** 2).sum(1))[:, None] * np.sqrt((wd ** 2).sum(1))[None, :]
    assert_close(Y[toks][:, rows], ref, bound, f"{m.name} n_tok={n_tok}")
    assert np.isfinite(Y).all()


@pytest.mark.parametrize("i", range(len(workloads.Q8_0_SQUARE)))
def test_full_q8_0_square(syn, i):
    sampled_check(syn, workloads.Q8_0_SQUARE[i], 1, 1, i, n_rows=2048)


@pytest.mark.parametrize("i", range(len(workloads.LLAMA1B_LAYER)))
def test_full_llama1b_layer_decode(syn, i):
    sampled_check(syn, workloads.LLAMA1B_LAYER[i], 1, 2, i, n_rows=512)


@pytest.mark.parametrize("n_tok", [1, 4])
def test_full_lm_head(syn, n_tok):
    sampled_check(syn, workloads.LM_HEAD_1B[0], n_tok, 3, 0, n_rows=96)


@pytest.mark.parametrize("i", range(len(workloads.LLAMA8B_FFN)))
def test_full_llama8b_ffn_prefill(syn, i):
    sampled_check(syn, workloads.LLAMA8B_FFN[i], 512, 4, i, n_rows=48, n_toks=6)


# the Llama-8B Q4_K_M sweep: one matrix of every distinct (format, shape) in the mix, as the
# decode product (1 token) and as the prefill product (2048 tokens), sampled entries
def _llama8b_distinct():
    mats = workloads.llama8b_q4_k_m()
    seen, picks = set(), []
    for i, m in enumerate(mats):
        key = (m.wtype, m.n_out, m.n_in)
        if key not in seen:
            seen.add(key)
            picks.append((i, m))
    return picks


LLAMA8B_DISTINCT = _llama8b_distinct()


@pytest.mark.parametrize("k", range(len(LLAMA8B_DISTINCT)))
def test_full_llama8b_sweep_decode(syn, k):
    i, m = LLAMA8B_DISTINCT[k]
    sampled_check(syn, m, 1, 5, i, n_rows=96, path="gemv")


@pytest.mark.parametrize("k", range(len(LLAMA8B_DISTINCT)))
def test_full_llama8b_sweep_prefill(syn, k):
    i, m = LLAMA8B_DISTINCT[k]
    sampled_check(syn, m, 2048, 5, i, n_rows=32, n_toks=4, path="gemm")


# Q4_0 / Q5_0 on the Llama-8B FFN up shape, as the benchmark runs them (decode inputs from
# workload 6, prefill inputs from workload 7)
@pytest.mark.parametrize("wt", [oracle.Q4_0, oracle.Q5_0])
def test_full_qx_0_decode(syn, wt):
    sampled_check(syn, workloads.Matrix("ffn_up", wt, 14336, 4096), 1, 6, 0, n_rows=256)


@pytest.mark.parametrize("wt", [oracle.Q4_0, oracle.Q5_0])
def test_full_qx_0_prefill(syn, wt):
    sampled_check(syn, workloads.Matrix("ffn_up", wt, 14336, 4096), 512, 7, 0, n_rows=48, n_toks=6)


# ----------------------------------------------------------------------------------------
# F16 weights (vec_dot_type F16): conversion bit-exact, products against the oracle
# ----------------------------------------------------------------------------------------

def test_f16_quantize_dequantize_bit_exact(syn):
    x = inputs_mixed(37, 520, 11)
    want = oracle.quantize(oracle.F16, x)
    got = host(syn.quantize(oracle.F16, dev(x)))
    assert np.array_equal(got, want)
    back = host(syn.dequantize(oracle.F16, dev(want), 520))
    assert np.array_equal(back.view(np.uint32), oracle.dequantize(oracle.F16, want, 520).view(np.uint32))
    with pytest.raises(syn.SynError):
        syn.quantize(oracle.F16, dev(np.full((1, 8), 1e6, np.float32)))


@pytest.mark.parametrize("shape", [(1, 8, 1), (77, 520, 1), (300, 2048, 3), (129, 4096, 8), (64, 1000, 40),
                                   (257, 768, 300), (128, 256, 16)])
@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_f16_mul_mat(syn, shape, path):
    n_out, n_in, n_tok = shape
    Y, ref, bound = run_mul_mat(syn, oracle.F16, n_out, n_in, n_tok, 3000 + n_out, path)
    assert_close(Y, ref, bound, f"f16 {shape} {path}")


def test_f16_in_a_batch(syn):
    items, refs = [], []
    for i, (wt, n_out, n_in) in enumerate([(oracle.F16, 100, 1024), (oracle.Q4_K, 64, 512), (oracle.F16, 33, 72)]):
        Wq = oracle.quantize(wt, synth.normal(700 + i, (n_out, n_in), 0.02))
        X = synth.normal(800 + i, (2, n_in))
        items.append((wt, dev(Wq), n_out, n_in, dev(X), torch.full((2, n_out), float("nan"), device="cuda")))
        refs.append((oracle.mul_mat(wt, Wq, n_out, n_in, X), tolerance(wt, Wq, n_in, X)))
    syn.mul_mat_batch(items, 2)
    for (wt, _, n_out, n_in, _, Yd), (ref, bound) in zip(items, refs):
        assert_close(host(Yd), ref, bound, f"batch {oracle.NAMES[wt]} {n_out}x{n_in}")
    assert syn.device_status() == syn.OK


@pytest.mark.parametrize("n_tok", [1, 512])
def test_full_f16(syn, n_tok):
    sampled_check(syn, workloads.Matrix("ffn_up", oracle.F16, 14336, 4096), n_tok, 8, 0, n_rows=96, n_toks=4,
                  path="gemv" if n_tok == 1 else "gemm")
