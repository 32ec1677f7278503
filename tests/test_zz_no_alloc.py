"""syn_mul_mat_prefill_static: the prefill product for callers that cannot allocate device
memory (fixed arenas, allocators or budgets that forbid cudaMalloc, paths that must not
let a library synchronize the device through cudaMalloc/cudaFree).  Its scratch is a
fixed device array inside the library.

Each product is checked through the C ABI against the CPU oracle, within the tolerance of
the parity tests (1e-4 * ||dequant(w_row)||_2 * ||x||_2 per element), on calls in a row
with different problems, so that every call after the first runs on scratch the one
before it left behind.  A product that fills the array exactly checks its last tokens
(the end of the array).  After the calls, syn_device_status reports no timeout.  Kept in a
file that pytest collects last.
"""
import numpy as np
import pytest

import oracle
from gguf_block_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 1e-4


@pytest.fixture(scope="module")
def syn():
    from gguf_block_quantized_gb300 import syn as s
    return s


def bound(wt, Wq, n_in, X):
    wd = oracle.dequantize(wt, Wq, n_in).astype(np.float64)
    return TOL * np.sqrt((X.astype(np.float64) ** 2).sum(1))[:, None] * np.sqrt((wd ** 2).sum(1))[None, :]


def static_prefill(syn, wt, Wd, n_out, n_in, Xd):
    Y = torch.full((Xd.shape[0], n_out), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = syn.syn_mul_mat_prefill_static(wt, Wd.data_ptr(), n_out, n_in, Xd.data_ptr(), Xd.shape[0],
                                        Y.data_ptr(), s)
    assert st == syn.OK, syn.syn_strerror(st)
    return Y


def check(Y, ref, bnd, what):
    assert np.isfinite(Y).all(), what
    err = np.abs(Y.astype(np.float64) - ref.astype(np.float64))
    assert (err <= bnd).all(), f"{what}: {(err > bnd).sum()} outside, max err/bound {(err / bnd).max():.3g}"


def test_static_scratch_matches_oracle_calls_in_a_row(syn):
    syn.device_status(True)
    cases = [(oracle.Q4_K, 1000, 2048, 300, 71), (oracle.Q6_K, 333, 1536, 40, 72),
             (oracle.Q8_0, 257, 1024, 130, 73), (oracle.F16, 200, 520, 77, 74),
             (oracle.Q4_K, 128, 512, 9, 75)]
    for wt, n_out, n_in, n_tok, seed in cases:
        W = oracle.quantize(wt, synth.normal(seed, (n_out, n_in), 0.02))
        X = synth.normal(seed + 100, (n_tok, n_in))
        got = static_prefill(syn, wt, torch.from_numpy(W).cuda(), n_out, n_in, torch.from_numpy(X).cuda())
        torch.cuda.synchronize()
        ref = oracle.mul_mat(wt, W, n_out, n_in, X)
        check(got.cpu().numpy(), ref, bound(wt, W, n_in, X), f"{oracle.NAMES[wt]} {n_out}x{n_in} n_tok={n_tok}")
    assert syn.device_status(True) == syn.OK


def test_static_scratch_at_exact_capacity(syn):
    """n_tok * n_in * 2 == the array's size: the last token's fp16 activations end at the
    array's last byte.  Sampled outputs (always the last tokens) against the oracle."""
    n_in = 4096
    n_tok = syn.STATIC_SCRATCH_BYTES // (2 * n_in)
    n_out = 160
    wt = oracle.Q4_K
    W = oracle.quantize(wt, synth.normal(81, (n_out, n_in), 0.02))
    X = synth.normal(82, (n_tok, n_in))
    got = static_prefill(syn, wt, torch.from_numpy(W).cuda(), n_out, n_in, torch.from_numpy(X).cuda())
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    rows = np.unique(np.concatenate([[0, n_out - 1], synth.integers(83, 24, 0, n_out)]))
    toks = np.unique(np.concatenate([[0, n_tok - 2, n_tok - 1], synth.integers(84, 8, 0, n_tok)]))
    ref = oracle.mul_mat_sampled(wt, W, n_out, n_in, X, rows, toks)
    check(got[toks][:, rows], ref, bound(wt, W[rows], n_in, X[toks]), "exact capacity")
    assert np.isfinite(got).all()
    assert syn.device_status(True) == syn.OK


def test_static_scratch_rejects_oversize_and_bad_shapes(syn):
    n_in = 4096
    n_tok = syn.STATIC_SCRATCH_BYTES // (2 * n_in) + 1
    p = 1 << 20
    assert syn.syn_mul_mat_prefill_static(oracle.Q4_K, p, 128, n_in, p, n_tok, p, None) == syn.ERR_TOO_LARGE
    assert syn.syn_strerror(syn.ERR_TOO_LARGE).decode().startswith("problem larger")
    # F16 rows are read 8 values at a time: n_in = 12 is rejected before anything is enqueued
    assert syn.syn_mul_mat_prefill_static(oracle.F16, p, 128, 12, p, 4, p, None) == syn.ERR_SHAPE
