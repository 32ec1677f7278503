"""Bounded device waits run out without hanging the GPU, and the library reports it.

Every wait of the decode and prefill kernels on an mbarrier is bounded: when it gives up
the kernel records SYN_ERR_TIMEOUT in a device word, stops the CTA's other threads, waits
for the copies and tensor-core operations it had already issued, frees its tensor memory
and returns.  To make those waits run out for certain, these tests load a checking build
of the library (libsyn_stall.so: the same sources compiled with SYN_TEST_STALL and a
20,000,000-cycle bound) in which the activation copies of the decode kernel and the
activation tiles of the prefill kernel are never issued, so the phases they would complete
never complete: a flag that nothing sets.  No GPU fault, trap or endless loop is involved.

Each stalled product must launch (SYN_OK), then syn_device_status must read SYN_ERR_TIMEOUT
once and SYN_OK after the clear.  Afterwards the normal library's products on the same
device still match the CPU oracle within the parity tolerance: the context is intact.
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
    stall = syn.bind(build.build(variant="stall"))
    return syn, stall


def _bound(wt, Wq, n_in, X):
    wd = oracle.dequantize(wt, Wq, n_in).astype(np.float64)
    return TOL * np.sqrt((X.astype(np.float64) ** 2).sum(1))[:, None] * np.sqrt((wd ** 2).sum(1))[None, :]


def _operands(wt, n_out, n_in, n_tok, seed):
    W = oracle.quantize(wt, synth.normal(seed, (n_out, n_in), 0.02))
    X = synth.normal(seed + 1, (n_tok, n_in))
    return W, X, torch.from_numpy(W).cuda(), torch.from_numpy(X).cuda()


def _expect_timeout(lib, syn, rc, what):
    assert rc == syn.OK, f"{what}: launch returned {lib.syn_strerror(rc).decode()}"
    st = lib.syn_device_status(1)
    assert st == syn.ERR_TIMEOUT, f"{what}: status {lib.syn_strerror(st).decode()} instead of a timeout"
    st = lib.syn_device_status(1)
    assert st == syn.OK, f"{what}: status not cleared ({lib.syn_strerror(st).decode()})"


# (format, n_out, n_in, n_tok): decode with a conversion launch (wide input), decode that
# converts inside its CTAs (narrow input), Q8_0 decode and prefill, prefill on one tile, on
# a K-split product, F16 weights
STALL_CASES = [
    (oracle.Q4_K, 512, 14336, 1),
    (oracle.Q6_K, 256, 1024, 2),
    (oracle.Q8_0, 300, 768, 3),
    (oracle.Q8_0, 300, 768, 11),
    (oracle.Q4_K, 256, 1024, 64),
    (oracle.Q6_K, 128, 8192, 40),
    (oracle.F16, 128, 256, 48),
]


@pytest.mark.parametrize("wt,n_out,n_in,n_tok", STALL_CASES)
def test_stalled_product_reports_timeout(libs, wt, n_out, n_in, n_tok):
    syn, stall = libs
    torch.cuda.set_device(0)
    stall.syn_device_status(1)
    _, _, Wd, Xd = _operands(wt, n_out, n_in, n_tok, 900 + n_in % 97)
    Y = torch.zeros((n_tok, n_out), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = stall.syn_mul_mat(wt, Wd.data_ptr(), n_out, n_in, Xd.data_ptr(), n_tok, Y.data_ptr(), s)
    _expect_timeout(stall, syn, rc, f"{oracle.NAMES[wt]} {n_out}x{n_in} n_tok={n_tok}")


def test_stalled_grouped_and_static_calls_report_timeout(libs):
    syn, stall = libs
    torch.cuda.set_device(0)
    stall.syn_device_status(1)
    s = torch.cuda.current_stream().cuda_stream
    # a grouped decode launch of three products
    ops = [_operands(wt, n_out, 2048, 1, 950 + k) for k, (wt, n_out) in
           enumerate([(oracle.Q4_K, 512), (oracle.Q6_K, 128), (oracle.Q4_K, 2048)])]
    Xd = ops[0][3]
    Ys = [torch.zeros((1, W.shape[0]), device="cuda") for W, _, _, _ in ops]
    descs = (syn.MatDesc * 3)()
    for k, ((W, _, Wd, _), wt) in enumerate(zip(ops, [oracle.Q4_K, oracle.Q6_K, oracle.Q4_K])):
        descs[k] = syn.MatDesc(wt, Wd.data_ptr(), W.shape[0], 2048, Xd.data_ptr(), Ys[k].data_ptr())
    rc = stall.syn_mul_mat_batch(3, ctypes.cast(descs, ctypes.POINTER(syn.MatDesc)), 1, s)
    _expect_timeout(stall, syn, rc, "grouped decode")
    # the prefill entry point that allocates nothing (its status word is in its fixed array)
    _, _, Wd, Xd = _operands(oracle.Q4_K, 256, 1024, 32, 960)
    Y = torch.zeros((32, 256), device="cuda")
    rc = stall.syn_mul_mat_prefill_static(oracle.Q4_K, Wd.data_ptr(), 256, 1024, Xd.data_ptr(), 32,
                                          Y.data_ptr(), s)
    _expect_timeout(stall, syn, rc, "static prefill")


def test_waitless_kernels_report_no_timeout(libs):
    """F16 decode has no mbarrier wait: the stall build runs it normally, and it matches the
    oracle."""
    syn, stall = libs
    torch.cuda.set_device(0)
    stall.syn_device_status(1)
    W, X, Wd, Xd = _operands(oracle.F16, 96, 512, 1, 970)
    Y = torch.zeros((1, 96), device="cuda")
    rc = stall.syn_mul_mat(oracle.F16, Wd.data_ptr(), 96, 512, Xd.data_ptr(), 1, Y.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    assert rc == syn.OK
    assert stall.syn_device_status(1) == syn.OK
    ref = oracle.mul_mat(oracle.F16, W, 96, 512, X)
    assert (np.abs(Y.cpu().numpy().astype(np.float64) - ref) <= _bound(oracle.F16, W, 512, X)).all()


def test_device_usable_after_timeouts(libs):
    """After the stalled launches, the normal library's decode and prefill products on the
    same device match the oracle and its own status word reads SYN_OK."""
    syn, stall = libs
    torch.cuda.set_device(0)
    s = torch.cuda.current_stream().cuda_stream
    _, _, Wd, Xd = _operands(oracle.Q4_K, 256, 1024, 64, 980)
    Y = torch.zeros((64, 256), device="cuda")
    rc = stall.syn_mul_mat(oracle.Q4_K, Wd.data_ptr(), 256, 1024, Xd.data_ptr(), 64, Y.data_ptr(), s)
    _expect_timeout(stall, syn, rc, "prefill before the normal products")
    for wt, n_out, n_in, n_tok, seed in [(oracle.Q4_K, 300, 2048, 1, 981), (oracle.Q6_K, 256, 1024, 5, 983),
                                         (oracle.Q4_K, 256, 1024, 64, 985), (oracle.Q8_0, 200, 768, 33, 987)]:
        W, X, Wd, Xd = _operands(wt, n_out, n_in, n_tok, seed)
        got = syn.mul_mat(wt, Wd, n_out, n_in, Xd).cpu().numpy().astype(np.float64)
        ref = oracle.mul_mat(wt, W, n_out, n_in, X)
        err = np.abs(got - ref)
        bnd = _bound(wt, W, n_in, X)
        assert (err <= bnd).all(), f"{oracle.NAMES[wt]} {n_out}x{n_in} n_tok={n_tok}: max err/bound {(err / bnd).max():.3g}"
    assert syn.device_status(True) == syn.OK
