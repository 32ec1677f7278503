"""syn_mul_mat_prefill_static: the prefill product for callers that cannot allocate device
memory (fixed arenas, allocators or budgets that forbid cudaMalloc, paths that must not
let a library synchronize the device through cudaMalloc/cudaFree).  Its scratch is a
fixed device array inside the library.

Checked through the C ABI against syn_mul_mat's own prefill path, within the tolerance of
the parity tests (1e-4 * ||dequant(w_row)||_2 * ||x||_2 per element), on two calls in a
row with different problems, so that the second call runs on scratch the first one left
behind.  Kept in a file that pytest collects last.
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


def existing_prefill(syn, wt, Wd, n_out, n_in, Xd):
    old = syn.set_gemv_max_tok(0)
    try:
        return syn.mul_mat(wt, Wd, n_out, n_in, Xd)
    finally:
        syn.set_gemv_max_tok(old)


def static_prefill(syn, wt, Wd, n_out, n_in, Xd):
    Y = torch.full((Xd.shape[0], n_out), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = syn.syn_mul_mat_prefill_static(wt, Wd.data_ptr(), n_out, n_in, Xd.data_ptr(), Xd.shape[0],
                                        Y.data_ptr(), s)
    assert st == syn.OK, syn.syn_strerror(st)
    return Y


def test_static_scratch_matches_existing_prefill_two_calls(syn):
    cases = [(oracle.Q4_K, 1000, 2048, 300, 71), (oracle.Q6_K, 333, 1536, 40, 72)]
    for wt, n_out, n_in, n_tok, seed in cases:
        W = oracle.quantize(wt, synth.normal(seed, (n_out, n_in), 0.02))
        X = synth.normal(seed + 100, (n_tok, n_in))
        Wd, Xd = torch.from_numpy(W).cuda(), torch.from_numpy(X).cuda()
        got = static_prefill(syn, wt, Wd, n_out, n_in, Xd)
        want = existing_prefill(syn, wt, Wd, n_out, n_in, Xd)
        torch.cuda.synchronize()
        got, want = got.cpu().numpy(), want.cpu().numpy()
        assert np.isfinite(got).all()
        err = np.abs(got.astype(np.float64) - want.astype(np.float64))
        assert (err <= bound(wt, W, n_in, X)).all(), f"case {(wt, n_out, n_in, n_tok)}: max err {err.max()}"


def test_static_scratch_rejects_oversize(syn):
    n_in = 4096
    n_tok = syn.STATIC_SCRATCH_BYTES // (2 * n_in) + 1
    p = 1 << 20
    assert syn.syn_mul_mat_prefill_static(oracle.Q4_K, p, 128, n_in, p, n_tok, p, None) == syn.ERR_TOO_LARGE
    assert syn.syn_strerror(syn.ERR_TOO_LARGE).decode().startswith("problem larger")
