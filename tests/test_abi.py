"""The C-ABI library: it builds, loads and exports every declared symbol,
and host-side argument checks reject bad calls before any GPU work (CPU)."""
import ctypes
import os
import re

import pytest

import graph_transformer_sparse_gb300 as gt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "gtattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gtattn_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    gt.build()
    return gt.load()


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("gtattn_csr_build", "gtattn_fwd", "gtattn_fwd_plan", "gtattn_fwd_probs",
                 "gtattn_coo_to_csr", "gtattn_csr_validate", "gtattn_status_string"):
        assert must in names
    assert set(names) == set(gt.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_checking_build_links_and_exports_every_declared_symbol():
    # the GTATTN_DEBUG build resolves every symbol it uses (loaded with
    # RTLD_NOW, no call is made) and exports the same boundary
    from graph_transformer_sparse_gb300 import _build
    path = _build.build(debug=True)
    dlib = ctypes.CDLL(path, mode=os.RTLD_NOW)
    for name in _declared():
        assert hasattr(dlib, name), name
    # (without a GPU every call stops at the host checks)
    fn = dlib.gtattn_status_string
    fn.restype = ctypes.c_char_p
    fn.argtypes = [ctypes.c_int]
    assert fn(gt.GTATTN_ERR_BAD_CSR)


def test_status_strings(lib):
    assert gt.gtattn_status_string(0) == "ok"
    assert gt.gtattn_status_string(2) == "malformed CSR"
    assert gt.gtattn_status_string(99) == "unknown status"


def test_host_argument_checks(lib):
    # rejected before any device work: no GPU needed
    INV = gt.GTATTN_ERR_INVALID_ARG
    f = lib.gtattn_fwd
    assert f(None, None, None, None, None, None, 4, 4, 2, 8, 1.0, 0, None) == INV      # null indptr
    assert f(16, 16, 16, 16, 16, 16, -1, 4, 2, 8, 1.0, 0, None) == INV                # N < 0
    assert f(16, 16, 16, 16, 16, 16, 4, 4, 0, 8, 1.0, 0, None) == INV                 # H < 1
    assert f(16, 16, 16, 16, 16, 16, 4, 4, 2, 1000, 1.0, 0, None) == INV              # H*D > 1024
    assert f(16, 16, 16, 16, 16, 16, 4, 4, 2, 8, 1.0, 7, None) == INV                 # dtype
    assert f(16, 16, 18, 16, 16, 16, 4, 4, 2, 8, 1.0, 0, None) == INV                 # misaligned f32
    assert f(16, 16, 16, None, 16, 16, 4, 4, 2, 8, 1.0, 0, None) == INV               # null K, nnz > 0
    assert f(16, 16, 16, 16, 16, 16, 1 << 31, 4, 2, 8, 1.0, 0, None) == INV           # N too large
    assert lib.gtattn_fwd_plan(None, 16, 16, 16, 16, 16, 16, 2, 8, 1.0, 0, None) == INV
    assert lib.gtattn_fwd_probs(16, 16, 16, 16, 16, 16, 18, 16, 4, 4, 2, 8, 1.0, 0, None) == INV
    assert lib.gtattn_csr_build(16, 16, 4, 4, None, None, None) == INV                 # null plan_out
    plan = ctypes.c_void_p()
    assert lib.gtattn_csr_build(16, 16, -3, 4, None, ctypes.byref(plan), None) == INV
    assert lib.gtattn_csr_validate(None, None, 3, 0, None) == INV
    assert lib.gtattn_coo_to_csr(None, None, 4, 4, 16, 16, None) == INV
    assert lib.gtattn_plan_destroy(None) == 0
    assert lib.gtattn_plan_get_info(None, None) == INV


def test_host_argument_checks_bias_weighted_bwd_ndh(lib):
    # the entry points beyond the plain forward, rejected before device work
    INV, OK = gt.GTATTN_ERR_INVALID_ARG, gt.GTATTN_OK
    fb = lib.gtattn_fwd_bias   # indptr indices Q K V bias out logits probs N nnz H D scale dtype stream
    assert fb(16, 16, 16, 16, 16, None, 16, None, None, 4, 4, 2, 8, 1.0, 0, None) == INV   # null bias, nnz > 0
    assert fb(16, 16, 16, 16, 16, 18, 16, None, None, 4, 4, 2, 8, 1.0, 0, None) == INV     # misaligned bias
    assert fb(None, 16, 16, 16, 16, 16, 16, None, None, 4, 4, 2, 8, 1.0, 0, None) == INV   # null indptr
    fw = lib.gtattn_fwd_weighted   # indptr indices values Q K V out logits probs N nnz H D scale dtype stream
    assert fw(16, 16, None, 16, 16, 16, 16, None, None, 4, 4, 2, 8, 1.0, 0, None) == INV   # null values
    assert fw(16, 16, 18, 16, 16, 16, 16, None, None, 4, 4, 2, 8, 1.0, 0, None) == INV     # misaligned values
    assert fw(16, 16, 16, 16, 16, 16, 16, None, None, 4, 4, 0, 8, 1.0, 0, None) == INV     # H < 1
    fg = lib.gtattn_bwd   # indptr indices Q K V dO dQ dK dV N nnz H D scale dtype stream
    assert fg(16, 16, 16, 16, 16, 16, 16, 16, 16, -1, 4, 2, 8, 1.0, 0, None) == INV        # N < 0
    assert fg(16, 16, 16, 16, 16, 16, 16, 16, 16, 4, 4, 200, 1, 1.0, 0, None) == INV       # H > 128
    assert fg(16, 16, 16, 16, 16, 16, 16, 16, 16, 4, 4, 2, 8, 1.0, 7, None) == INV         # dtype
    assert fg(16, 16, 16, 16, 16, 16, None, 16, 16, 4, 4, 2, 8, 1.0, 0, None) == INV       # null dQ
    assert fg(16, 16, 16, 16, 16, 18, 16, 16, 16, 4, 4, 2, 8, 1.0, 0, None) == INV         # misaligned dO
    assert fg(16, 18, 16, 16, 16, 16, 16, 16, 16, 4, 4, 2, 8, 1.0, 0, None) == INV         # misaligned indices
    assert fg(16, 16, 16, None, 16, 16, 16, 16, 16, 4, 4, 2, 8, 1.0, 0, None) == INV       # null K, nnz > 0
    assert fg(None, 16, 16, 16, 16, 16, 16, 16, 16, 4, 4, 2, 8, 1.0, 0, None) == INV       # null indptr
    assert fg(16, None, None, None, None, None, None, None, None, 0, 0, 2, 8, 1.0, 0, None) == OK   # N = 0
    fp = lib.gtattn_bwd_plan   # plan indptr indices Q K V O stats dO dQ dK dV H D scale dtype stream
    assert fp(None, 16, 16, 16, 16, 16, None, None, 16, 16, 16, 16, 2, 8, 1.0, 0, None) == INV     # null plan
    assert fp(None, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 2, 8, 1.0, 0, None) == INV         # null plan
    fs = lib.gtattn_fwd_plan_stats   # plan indptr indices Q K V out stats H D scale dtype stream
    assert fs(None, 16, 16, 16, 16, 16, 16, 16, 2, 8, 1.0, 0, None) == INV                 # null plan
    assert fs(16, 16, 16, 16, 16, 16, 16, None, 2, 8, 1.0, 0, None) == INV                 # null stats
    assert fs(16, 16, 16, 16, 16, 16, 16, 18, 2, 8, 1.0, 0, None) == INV                   # misaligned stats
    fn = lib.gtattn_fwd_ndh   # indptr indices Q K V out N nnz H D scale dtype stream
    assert fn(None, 16, 16, 16, 16, 16, 4, 4, 2, 8, 1.0, 0, None) == INV                   # null indptr
    assert fn(16, 16, 16, 16, 16, 16, 4, 4, 2, 1000, 1.0, 0, None) == INV                  # H*D > 1024
    assert fn(16, 16, 16, 16, 16, None, 4, 4, 2, 8, 1.0, 0, None) == INV                   # null out


def test_host_argument_checks_proj(lib):
    # gtattn_fwd_proj and gtattn_device_errors, rejected before device work
    INV, OK = gt.GTATTN_ERR_INVALID_ARG, gt.GTATTN_OK
    f = lib.gtattn_fwd_proj   # indptr indices X Wqkv bqkv Wo bo Y qkv attn N nnz F_in H D F_out heads_inner scale dtype stream
    assert f(None, 16, 16, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 0, None) == INV  # null indptr
    assert f(16, 16, None, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 0, None) == INV  # null X
    assert f(16, 16, 16, 16, None, None, None, 16, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 0, None) == INV  # null Wo
    assert f(16, 16, 16, 16, None, 16, None, 16, None, None, 4, 4, 0, 2, 4, 8, 0, 1.0, 0, None) == INV    # F_in 0
    assert f(16, 16, 16, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 4, 0, 0, 1.0, 0, None) == INV    # F_out 0
    assert f(16, 16, 16, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 600, 8, 0, 1.0, 0, None) == INV  # H*D
    assert f(16, 16, 16, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 3, 1.0, 0, None) == INV    # heads_inner
    assert f(16, 16, 16, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 9, None) == INV    # dtype
    assert f(16, 16, 18, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 0, None) == INV    # fp32 X
    assert f(16, 16, 16, 16, 18, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 0, None) == INV     # bias
    assert f(16, 16, 16, 16, None, 16, None, 17, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 1, None) == INV    # bf16 Y
    assert f(16, 16, None, None, None, None, None, None, None, None, 0, 0, 8, 2, 4, 8, 0, 1.0, 0, None) == OK
    assert lib.gtattn_device_errors(None, 0) == INV


def test_product_path_has_no_oracle_dependency():
    # the package and its sources never import or link the oracle
    pkg = os.path.join(ROOT, "graph_transformer_sparse_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in text.lower(), f"{fn} mentions the oracle"
