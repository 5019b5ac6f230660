"""The C-ABI library loads and exports every symbol include/mxmoe.h declares (no GPU calls)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"MX_API\s+[\w\s\*]+?\b(\w+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from mxfp8_block_scaled_rowwise_gb300 import _build, binding
    _build.build()
    return binding.load()


def test_header_declares_the_path():
    d = _declared()
    for name in ("mxfp8_quantize", "moe_permute", "grouped_gemm_mxfp8_fwd", "grouped_gemm_mxfp8_dgrad",
                 "grouped_gemm_mxfp8_wgrad"):
        assert name in d


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_host_only_helpers(lib):
    from mxfp8_block_scaled_rowwise_gb300 import binding as mx
    assert mx.mx_sf_bytes(1, 1) == 128 * 4
    assert mx.mx_sf_bytes(16384, 224) == 16384 * 224
    assert mx.mx_sf_bytes(130, 7) == 256 * 8
    assert mx.mx_sf_bytes_x4(130, 7) == 4 * 256 * 8
    assert mx.mx_sf_bytes_x4(-1, 7) == 0
    assert mx.mx_padded_rows_bound(131072, 32) == 131072 + 4096
    assert mx.mx_padded_rows_bound(0, 4) == 512
    assert lib.mx_status_str(-2) == b"MX_ERR_ALIGNMENT"
    assert mx.moe_permute_workspace_bytes(4096, 8, 128) >= 2 * 16 * 128 * 4


def test_argument_validation_needs_no_gpu(lib):
    # invalid arguments are rejected on the host before any CUDA call
    assert lib.mxfp8_quantize(None, 10, 33, 1, None, None, 0, 0, None, None, None, None, None, None) == -1
    assert lib.mxfp8_quantize(None, 10, 32, 4, None, None, 0, 0, None, None, None, None, None, None) == -1
    # mode bits: an _X4 bit needs its form; unknown bits are rejected (checked before the pointers)
    for bad in (4, 8, 1 | 8, 2 | 4, 64, 3 | 64, 0):
        assert lib.mxfp8_quantize(16, 128, 32, bad, None, None, 0, 128, 16, 16, 16, 16, None, None) == -1, bad
        assert lib.mxfp8_swiglu_quantize(16, 128, 128, bad, None, None, 0, 128, 16, 16, 16, 16, None, None) == -1, bad


def test_blocked_layout_argument_validation(lib):
    # mxfp8_quantize(x, rows, cols, mode, seg_off, seg_poff, nseg, ld_col, q_row, sf_row, q_col, sf_col, err, s):
    # a _BLK bit needs its form; the blocked rowwise form whole 128 x 128 blocks and no segments,
    # the blocked columnwise form cols % 128 == 0; only mxfp8_quantize(_ex) writes blocked codes
    from mxfp8_block_scaled_rowwise_gb300 import binding as mx
    q = lib.mxfp8_quantize
    RB, CB = mx.MX_ROWWISE_BLK, mx.MX_COLWISE_BLK
    assert (RB, CB, mx.MX_GEMM_B_BLOCKED) == (16, 32, 2)
    for bad in (RB, CB, 1 | CB, 2 | RB, 3 | RB | 4 | 64):
        assert q(16, 256, 256, bad, None, None, 0, 256, 16, 16, 16, 16, None, None) == -1, bad
    assert q(16, 256, 96, 1 | RB, None, None, 0, 256, 16, 16, 16, 16, None, None) == -1      # cols % 128
    assert q(16, 200, 256, 1 | RB, None, None, 0, 256, 16, 16, 16, 16, None, None) == -1     # rows % 128
    assert q(16, 256, 256, 1 | RB, 16, 16, 2, 512, 16, 16, 16, 16, None, None) == -1         # segments
    assert q(16, 200, 96, 2 | CB, None, None, 0, 256, 16, 16, 16, 16, None, None) == -1      # cols % 128
    assert lib.mxfp8_swiglu_quantize(16, 128, 128, 1 | RB, None, None, 0, 128, 16, 16, 16, 16, None, None) == -1
    assert lib.mxfp8_gather_quantize(16, 128, 128, 2 | CB, 16, 16, 16, 1, 128, 128, 16, 16, 16, 16, 16,
                                     None) == -1
    # GEMM flags: bits other than MX_GEMM_B_SCALES_X1 | MX_GEMM_B_BLOCKED are rejected on the host
    f = lib.grouped_gemm_mxfp8_fwd_ex
    assert f(16, 16, 16, 16, 16, 16, 4, 16, 128, 128, 16, 4, 16, None) == -1
    assert f(16, 16, 16, 16, 16, 16, 4, 16, 100, 128, 16, 2, 16, None) == -3                 # N % 128 still
    assert lib.grouped_gemm_mxfp8_fwd(1, 1, 1, 1, 1, 1, 4, 16, 100, 128, 1, 1, None) == -3   # N % 128
    assert lib.grouped_gemm_mxfp8_fwd(16, 16, 16, 16, 16, 16, 4, 16, 128, 128, 8, 16, None) == -2  # misaligned C
    assert lib.moe_permute(None, 4, 0, 4, None, None, None, None, None, None, None, 0, None, None, None, 0, None,
                           None) == -1


def test_fused_swiglu_gemm_argument_validation(lib):
    # grouped_gemm_mxfp8_fwd_swiglu(A, SFA, W1, SFW1, off, poff, E, R, I, K, out1, h_qrow, h_sfrow,
    #                               h_qcol, h_sfcol, ld_col, h_mode, dev_err, stream)
    f = lib.grouped_gemm_mxfp8_fwd_swiglu
    ok = [16] * 6
    outs = [16] * 5
    R, E = 300, 4
    ld = 300 + 127 * 4 + (-(300 + 127 * 4)) % 128          # the padded-position bound
    m = 3 | 8                                                                 # h_mode: both forms, columnwise x4
    assert f(*ok, E, R, 200, 384, *outs, ld, m, 16, None) == -3              # I % 128
    assert f(*ok, E, R, 256, 100, *outs, ld, m, 16, None) == -3              # K % 128
    assert f(*ok, E, R, 256, 384, *outs, ld - 128, m, 16, None) == -1        # ld_col below the bound
    assert f(*ok, E, R, 256, 384, *outs, ld + 64, m, 16, None) == -1         # ld_col % 128
    assert f(*ok, 0, R, 256, 384, *outs, ld, m, 16, None) == -1              # E
    assert f(None, *ok[1:], E, R, 256, 384, *outs, ld, m, 16, None) == -1    # missing A
    assert f(*ok, E, R, 256, 384, 16, 16, 16, 16, 8, ld, m, 16, None) == -2  # misaligned h_sfcol
    assert f(*ok, E, R, 256, 384, *outs, ld, m, None, None) == -1            # dev_err required
    for bad in (1, 2, 1 | 4, 3 | 16):                                        # both forms required; no unknown bits
        assert f(*ok, E, R, 256, 384, *outs, ld, bad, 16, None) == -1, bad
