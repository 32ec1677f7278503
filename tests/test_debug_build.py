"""The SYN_DEBUG build: index checks in every kernel, the stand-in for a memory checker.

libsyn_debug.so is the library compiled with SYN_DEBUG: before each access its kernels
check the indices and copy windows they derive from the launch geometry (weight-stage
windows against the slot and against W, TMA coordinates and their 16-byte alignment,
shared-memory activation areas, tile and unit coordinates, output indices).  A failed
check records the failure, skips the access, and syn_device_status returns SYN_ERR_BOUNDS.

First the checks are shown to be compiled in (one deliberately out-of-range check, whose
guarded store is skipped, reads back as SYN_ERR_BOUNDS).  Then small products with the
awkward geometries run through it and must leave every check passing while matching the
CPU oracle: ragged row and token tiles, 34- and 210-byte blocks ending mid-word at the end
of W, rows whose pitch is not a multiple of 16 bytes (per-row copy windows), products split
along K, a grouped decode launch, and the quantizers (bit-exact).
"""
import ctypes

import numpy as np
import pytest

import oracle
from gguf_block_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 1e-4


@pytest.fixture(scope="module")
def libs():
    from gguf_block_quantized_gb300 import build, syn
    dbg = syn.bind(build.build(variant="debug"))
    torch.cuda.set_device(0)
    dbg.syn_device_status(1)
    return syn, dbg


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _status(syn, dbg):
    st = dbg.syn_device_status(1)
    return st, dbg.syn_strerror(st).decode()


def _bound(wt, Wq, n_in, X):
    wd = oracle.dequantize(wt, Wq, n_in).astype(np.float64)
    return TOL * np.sqrt((X.astype(np.float64) ** 2).sum(1))[:, None] * np.sqrt((wd ** 2).sum(1))[None, :]


def test_checks_are_compiled_in(libs):
    syn, dbg = libs
    assert syn.syn_debug_bounds_selftest(_stream()) == 1, "the product build has no index checks"
    assert dbg.syn_debug_bounds_selftest(_stream()) == syn.OK
    assert _status(syn, dbg)[0] == syn.ERR_BOUNDS
    assert _status(syn, dbg)[0] == syn.OK, "status not cleared"


# (format, n_out, n_in, n_tok)
PRODUCTS = [
    # decode
    (oracle.Q8_0, 301, 800, 1),    # 25 x 34-byte blocks per row: pitch 850, W ends mid-word
    (oracle.Q6_K, 131, 768, 3),    # 630-byte rows
    (oracle.Q4_K, 257, 2048, 1),
    (oracle.Q4_K, 96, 14336, 2),   # rows of 56 blocks, several stages per row
    (oracle.Q6_K, 203, 2048, 4),   # two rows of 8 blocks per warp step, an odd row count
    (oracle.Q4_0, 129, 544, 1),
    (oracle.Q5_0, 67, 544, 4),
    (oracle.F16, 97, 264, 2),
    # prefill
    (oracle.Q4_K, 300, 1024, 77),  # ragged row and token tiles
    (oracle.Q6_K, 131, 768, 40),   # per-row copy windows (pitch 630), elementwise epilogue
    (oracle.Q8_0, 130, 800, 50),   # per-row windows, partial last 256-k step
    (oracle.Q4_K, 128, 8192, 40),  # split along K: reduce-adds into a zeroed Y
    (oracle.Q6_K, 2048, 2048, 300),  # several waves of tiles
    (oracle.Q4_0, 200, 512, 33),
    (oracle.Q5_0, 129, 544, 20),
    (oracle.F16, 130, 264, 50),
]


@pytest.mark.parametrize("wt,n_out,n_in,n_tok", PRODUCTS)
def test_products_pass_every_check(libs, wt, n_out, n_in, n_tok):
    syn, dbg = libs
    seed = 3000 + 7 * n_out + n_in % 101 + n_tok
    W = oracle.quantize(wt, synth.normal(seed, (n_out, n_in), 0.02))
    X = synth.normal(seed + 1, (n_tok, n_in))
    Wd, Xd = torch.from_numpy(W).cuda(), torch.from_numpy(X).cuda()
    Y = torch.full((n_tok, n_out), float("nan"), device="cuda")
    rc = dbg.syn_mul_mat(wt, Wd.data_ptr(), n_out, n_in, Xd.data_ptr(), n_tok, Y.data_ptr(), _stream())
    assert rc == syn.OK, dbg.syn_strerror(rc).decode()
    st, msg = _status(syn, dbg)
    assert st == syn.OK, msg
    got = Y.cpu().numpy().astype(np.float64)
    ref = oracle.mul_mat(wt, W, n_out, n_in, X)
    err = np.abs(got - ref)
    bnd = _bound(wt, W, n_in, X)
    assert np.isfinite(got).all() and (err <= bnd).all(), f"max err/bound {(err / bnd).max():.3g}"


def test_grouped_decode_passes_every_check(libs):
    syn, dbg = libs
    n_in = 2048
    shapes = [(oracle.Q4_K, 512), (oracle.Q6_K, 131), (oracle.Q4_K, 2048), (oracle.Q6_K, 2048)]
    X = synth.normal(3100, (1, n_in))
    Xd = torch.from_numpy(X).cuda()
    Ws = [oracle.quantize(wt, synth.normal(3101 + k, (n_out, n_in), 0.02)) for k, (wt, n_out) in enumerate(shapes)]
    Wds = [torch.from_numpy(w).cuda() for w in Ws]
    Ys = [torch.full((1, n_out), float("nan"), device="cuda") for _, n_out in shapes]
    descs = (syn.MatDesc * len(shapes))()
    for k, (wt, n_out) in enumerate(shapes):
        descs[k] = syn.MatDesc(wt, Wds[k].data_ptr(), n_out, n_in, Xd.data_ptr(), Ys[k].data_ptr())
    rc = dbg.syn_mul_mat_batch(len(shapes), ctypes.cast(descs, ctypes.POINTER(syn.MatDesc)), 1, _stream())
    assert rc == syn.OK
    st, msg = _status(syn, dbg)
    assert st == syn.OK, msg
    for k, (wt, n_out) in enumerate(shapes):
        got = Ys[k].cpu().numpy().astype(np.float64)
        ref = oracle.mul_mat(wt, Ws[k], n_out, n_in, X)
        assert (np.abs(got - ref) <= _bound(wt, Ws[k], n_in, X)).all(), f"product {k}"


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_K, oracle.Q6_K, oracle.Q8_K, oracle.Q4_0, oracle.Q5_0,
                                oracle.F16])
def test_quantize_dequantize_pass_every_check(libs, wt):
    syn, dbg = libs
    n_rows, n_in = 37, 1024
    W = synth.normal(3200 + wt, (n_rows, n_in), 0.02)
    Wd = torch.from_numpy(W).cuda()
    nbytes = n_rows * (n_in // syn.BLOCK_ELEMS[wt]) * syn.BLOCK_BYTES[wt]
    q = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert dbg.syn_quantize(wt, Wd.data_ptr(), q.data_ptr(), n_rows, n_in, _stream()) == syn.OK
    back = torch.empty((n_rows, n_in), device="cuda")
    assert dbg.syn_dequantize(wt, q.data_ptr(), back.data_ptr(), n_rows, n_in, _stream()) == syn.OK
    st, msg = _status(syn, dbg)
    assert st == syn.OK, msg
    ref = oracle.quantize(wt, W)
    assert np.array_equal(q.cpu().numpy(), ref.reshape(-1))
    assert np.array_equal(back.cpu().numpy(), oracle.dequantize(wt, ref, n_in))
