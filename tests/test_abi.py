"""The C-ABI library builds, loads and exports every symbol include/syn.h declares; the
host-side argument checks answer without touching a GPU.  CPU only."""
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "syn.h")


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401  (loads the CUDA runtime libsyn links against)
    from gguf_block_quantized_gb300 import build
    build.build()
    from gguf_block_quantized_gb300 import syn
    return syn


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SYN_API\s+[\w\s\*]+?\b(syn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared()
    for must in ("syn_quantize", "syn_dequantize", "syn_mul_mat", "syn_quantize_activations",
                 "syn_block_elems", "syn_block_bytes", "syn_row_bytes", "syn_strerror"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (syn_\w+)", out))
    missing = [n for n in declared() if n not in exported]
    assert not missing, missing
    assert {n for n, _, _ in lib.EXPORTS} == set(declared())


@pytest.mark.parametrize("variant", ["debug", "stall"])
def test_checking_variants_build_and_export_the_boundary(lib, variant):
    """The index-check build and the timeout-test build compile here (cross-compiled for
    sm_103a) and export the same entry points; the product build says it has no checks."""
    from gguf_block_quantized_gb300 import build
    path = build.build(variant=variant)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (syn_\w+)", out))
    assert set(declared()) <= exported
    assert lib.syn_debug_bounds_selftest(None) == 1


def test_host_functions(lib):
    assert [lib.syn_block_elems(t) for t in (1, 2, 3, 4)] == [32, 256, 256, 256]
    assert [lib.syn_block_bytes(t) for t in (1, 2, 3, 4)] == [34, 144, 210, 292]
    assert lib.syn_block_elems(9) == -1 and lib.syn_block_bytes(0) == -1
    assert lib.syn_row_bytes(2, 4096) == 16 * 144
    assert lib.syn_row_bytes(3, 100) == -1 and lib.syn_row_bytes(1, 0) == -1
    assert lib.syn_strerror(lib.ERR_ALIGN).decode().startswith("pointer")
    old = lib.syn_set_gemv_max_tok(5)
    if not os.environ.get("SYN_GEMV_MAX_TOK"):
        assert old == -1  # per-format thresholds by default
    assert lib.syn_set_gemv_max_tok(old) == 5
    assert lib.syn_set_gemv_max_tok(-7) == old and lib.syn_set_gemv_max_tok(old) == -1
    assert lib.syn_set_deterministic(7) == 0 and lib.syn_set_deterministic(0) == 1
    assert lib.syn_set_sm_limit(-1) == -1
    assert lib.syn_set_sm_limit(5) == 0 and lib.syn_set_sm_limit(0) == 5
    old = lib.syn_set_prefill_expand_tok(0)
    if not os.environ.get("SYN_PREFILL_EXPAND_TOK"):
        assert old == 1536
    assert lib.syn_set_prefill_expand_tok(-3) == 0 and lib.syn_set_prefill_expand_tok(old) == 1536


def test_argument_checks_need_no_gpu(lib):
    L = lib
    p = 1 << 20  # any aligned non-null value: the checks below reject before any use
    assert L.syn_mul_mat(4, p, 4, 256, p, 1, p, None) == L.ERR_TYPE      # Q8_K weights
    assert L.syn_mul_mat(8, p, 4, 256, p, 1, p, None) == L.ERR_TYPE  # unknown format
    assert L.syn_mul_mat(2, p, 4, 100, p, 1, p, None) == L.ERR_SHAPE
    assert L.syn_mul_mat(2, p, 0, 256, p, 1, p, None) == L.ERR_SHAPE
    assert L.syn_mul_mat(2, p, 4, 256, p, -1, p, None) == L.ERR_SHAPE
    assert L.syn_mul_mat(2, p, 4, 256, p, 0, p, None) == L.OK           # no-op
    assert L.syn_mul_mat(2, None, 4, 256, p, 1, p, None) == L.ERR_NULL
    assert L.syn_mul_mat(2, p + 4, 4, 256, p, 1, p, None) == L.ERR_ALIGN
    assert L.syn_quantize(2, p, p, 1, 255, None) == L.ERR_SHAPE
    assert L.syn_quantize(8, p, p, 1, 256, None) == L.ERR_TYPE  # unknown format
    assert L.syn_mul_mat(7, p, 4, 100, p, 1, p, None) == L.ERR_SHAPE  # F16 rows: n_in % 8
    assert L.syn_quantize_activations(7, p, 1, 256, p, p, p, None) == L.ERR_TYPE  # F16: no integer form
    assert L.syn_quantize(1, p, p, 0, 32, None) == L.OK
    assert L.syn_quantize(1, p + 8, p, 1, 32, None) == L.ERR_ALIGN
    assert L.syn_dequantize(3, None, p, 1, 256, None) == L.ERR_NULL
    assert L.syn_dequantize_f16(1, p, p, 1, 256, None) == L.ERR_TYPE   # Q8_0: K-quants only
    assert L.syn_dequantize_f16(2, p, p, 1, 100, None) == L.ERR_SHAPE
    assert L.syn_dequantize_f16(3, None, p, 1, 256, None) == L.ERR_NULL
    assert L.syn_dequantize_f16(2, p + 2, p, 1, 256, None) == L.ERR_ALIGN
    assert L.syn_dequantize_f16(2, p, p, 0, 256, None) == L.OK
    assert L.syn_quantize_activations(4, p, 1, 256, p, p, p, None) == L.ERR_TYPE
    assert L.syn_quantize_activations(2, p, 1, 256, p, p, None, None) == L.ERR_NULL
    assert L.syn_block_sums(2, p, 1, 300, p, 1, p, None) == L.ERR_SHAPE


def test_staged_batch_checks_need_no_gpu(lib):
    """The host-staged grouped call rejects bad arguments before enqueuing any copy."""
    L = lib
    p = 1 << 20
    d = (L.MatDesc * 1)(L.MatDesc(2, p, 4, 256, p, p))
    bad = (L.MatDesc * 1)(L.MatDesc(2, p, 4, 100, p, p))  # n_in not a multiple of 256
    assert L.syn_mul_mat_batch_staged(1, bad, 1, p, p, 1024, p, p, 16, None) == L.ERR_SHAPE
    assert L.syn_mul_mat_batch_staged(1, d, 1, None, p, 1024, p, p, 16, None) == L.ERR_NULL
    assert L.syn_mul_mat_batch_staged(1, d, 1, p, p, 1024, p, None, 16, None) == L.ERR_NULL
    assert L.syn_mul_mat_batch_staged(1, d, -1, p, p, 1024, p, p, 16, None) == L.ERR_SHAPE
    assert L.syn_mul_mat_batch_staged(0, None, 1, None, None, 0, None, None, 0, None) == L.OK  # nothing to do


def test_prepared_batch_staging_sizes_checked(lib):
    """prepare_batch(..., staged=...) checks the staging buffers against their host
    counterparts when it is built (marshalling only: nothing is called)."""
    import torch
    W = torch.zeros(16 * 144 // 4, dtype=torch.int32)  # one Q4_K row of 4096 values, as bytes
    X, Y = torch.zeros(4096), torch.zeros(1)
    items = [(lib.Q4_K, W, 1, 4096, X, Y)]
    xh, yh = torch.zeros(4096), torch.zeros(1)
    with pytest.raises(ValueError):
        lib.PreparedBatch(items, 1, stream=0, staged=(xh, torch.zeros(100), Y, yh))
    with pytest.raises(ValueError):
        lib.PreparedBatch(items, 1, stream=0, staged=(xh, X, torch.zeros(0), yh))
    pb = lib.PreparedBatch(items, 1, stream=0, staged=(xh, X, Y, yh))
    assert pb._sargs[2] == 4096 * 4 and pb._sargs[5] == 4
