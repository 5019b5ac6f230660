"""Thin Python binding of the C ABI in include/mxmoe.h (argument marshalling only).

The raw functions carry the C names (``mxfp8_quantize``, ``moe_permute``,
``moe_gather_rows``, ``grouped_gemm_mxfp8_fwd`` / ``_dgrad`` / ``_wgrad``) and
take torch CUDA tensors for the pointer arguments; every step runs in the CUDA
library.  PyTorch provides device memory and the current stream only.  If the
library is missing, every call raises: there is no CPU fallback.

The ``*_alloc`` helpers below additionally allocate the output tensors with
torch (sizes from the C-ABI size helpers) before calling the raw function.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

MX_ROWWISE = 1
MX_COLWISE = 2
MX_ROWWISE_X4 = 4   # rowwise scales in the four-copy layout (B operands of the grouped GEMMs)
MX_COLWISE_X4 = 8   # columnwise scales in the four-copy layout
MX_ROWWISE_BLK = 16   # rowwise codes in the blocked code layout (128 x 128 blocks of 16 KiB)
MX_COLWISE_BLK = 32   # columnwise codes in the blocked code layout
MX_DTYPE_BF16 = 0
MX_DTYPE_F32 = 1
MX_SCALE_FLOOR = 0
MX_SCALE_RCEIL = 1
MX_DEVERR_BAD_EXPERT_ID = 1
MX_DEVERR_TIMEOUT = 2
MX_DEVERR_BAD_SEGMENTS = 4
MX_GEMM_B_SCALES_X1 = 1   # *_ex GEMM flag: B-operand scales in the plain one-copy layout
MX_GEMM_B_BLOCKED = 2     # *_ex GEMM flag: B-operand codes in the blocked code layout
MX_TESTING_FWD, MX_TESTING_DGRAD, MX_TESTING_WGRAD = 0, 1, 2


class TestingGemmOptions(ctypes.Structure):
    """mx_testing_gemm_options of include/mxmoe_testing.h (tests and A/B measurements only)."""
    _fields_ = [("ctas_per_mma", ctypes.c_int), ("wait_limit_ns", ctypes.c_uint64),
                ("withhold_operands", ctypes.c_int), ("raster_group", ctypes.c_int), ("cluster_pairs", ctypes.c_int)]

_lib = None


class MxError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libmxmoe.so (raise if it is missing and building is not requested)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise MxError("CUDA library %s is not built; run __graft_entry__.build()" % _build.LIB)
        _build.build()
    L = ctypes.CDLL(_build.LIB)
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sig = {
        "mx_sf_bytes": (sz, [i64, i64]),
        "mx_sf_bytes_x4": (sz, [i64, i64]),
        "mx_padded_rows_bound": (i64, [i64, i64]),
        "mxfp8_quantize": (i32, [P, i64, i64, i32, P, P, i32, i64, P, P, P, P, P, P]),
        "mxfp8_quantize_ex": (i32, [P, i32, i32, i64, i64, i32, P, P, i32, i64, P, P, P, P, P, P]),
        "mxfp8_swiglu_quantize": (i32, [P, i64, i64, i32, P, P, i32, i64, P, P, P, P, P, P]),
        "mxfp8_swiglu_bwd_quantize": (i32, [P, P, i64, i64, i32, P, P, i32, i64, P, P, P, P, P, P]),
        "mxfp8_gather_quantize": (i32, [P, i64, i64, i32, P, P, P, i32, i64, i64, P, P, P, P, P, P]),
        "moe_permute_workspace_bytes": (sz, [i64, i32, i32]),
        "moe_permute": (i32, [P, i64, i32, i32, P, P, P, P, P, P, P, i64, P, P, P, sz, P, P]),
        "moe_gather_rows": (i32, [P, i64, P, i64, P, P]),
        "moe_permute_noalloc": (i32, [P, i64, i32, i32, P, P, P, P, P, P, P, i64, P, P, P, P]),
        "moe_combine_fwd": (i32, [P, P, P, i64, i32, i64, i64, P, P, P]),
        "moe_combine_bwd": (i32, [P, P, P, P, i64, i32, i64, i64, P, P, P, P]),
        "moe_combine_bwd_ex": (i32, [P, P, P, P, i64, i32, i64, i64, P, P, P, P, P]),
        "mxfp8_gather_quantize_ex": (i32, [P, i64, i64, i32, P, P, P, P, i32, i64, i64, P, P, P, P, P, P]),
        "grouped_gemm_mxfp8_fwd": (i32, [P, P, P, P, P, P, i32, i64, i64, i64, P, P, P]),
        "grouped_gemm_mxfp8_fwd_swiglu": (i32, [P, P, P, P, P, P, i32, i64, i64, i64, P, P, P, P, P, i64, i32, P, P]),
        "grouped_gemm_mxfp8_dgrad": (i32, [P, P, P, P, P, P, i32, i64, i64, i64, P, P, P]),
        "grouped_gemm_mxfp8_wgrad": (i32, [P, P, P, P, P, P, i32, i64, i64, i64, P, P, P]),
        "grouped_gemm_mxfp8_fwd_ex": (i32, [P, P, P, P, P, P, i32, i64, i64, i64, P, i32, P, P]),
        "grouped_gemm_mxfp8_fwd_swiglu_ex": (i32, [P, P, P, P, P, P, i32, i64, i64, i64, P, P, P, P, P, i64, i32, i32,
                                                   P, P]),
        "grouped_gemm_mxfp8_dgrad_ex": (i32, [P, P, P, P, P, P, i32, i64, i64, i64, P, i32, P, P]),
        "grouped_gemm_mxfp8_wgrad_ex": (i32, [P, P, P, P, P, P, i32, i64, i64, i64, P, i32, P, P]),
        "mx_testing_grouped_gemm": (i32, [i32, P, P, P, P, P, P, i32, i64, i64, i64, i64, P, i32,
                                          ctypes.POINTER(TestingGemmOptions), P, P]),
        "mx_status_str": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def exported_symbols():
    return ["mx_sf_bytes", "mx_sf_bytes_x4", "mx_padded_rows_bound", "mxfp8_quantize", "mxfp8_quantize_ex", "mxfp8_gather_quantize",
            "mxfp8_swiglu_quantize", "mxfp8_swiglu_bwd_quantize", "moe_permute_workspace_bytes", "moe_permute",
            "moe_gather_rows", "moe_permute_noalloc", "moe_combine_fwd", "moe_combine_bwd", "grouped_gemm_mxfp8_fwd",
            "grouped_gemm_mxfp8_fwd_swiglu", "grouped_gemm_mxfp8_dgrad", "grouped_gemm_mxfp8_wgrad",
            "grouped_gemm_mxfp8_fwd_ex", "grouped_gemm_mxfp8_fwd_swiglu_ex", "grouped_gemm_mxfp8_dgrad_ex",
            "grouped_gemm_mxfp8_wgrad_ex", "mx_testing_grouped_gemm", "moe_combine_bwd_ex", "mxfp8_gather_quantize_ex",
            "mx_status_str"]


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    assert t.is_cuda and t.is_contiguous(), "device tensors must be contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, what: str):
    if status != 0:
        raise MxError("%s failed: %s (%d)" % (what, load().mx_status_str(status).decode(), status))


# ------------------------------------------------------------------ size helpers
def mx_sf_bytes(rows: int, kb: int) -> int:
    return int(load().mx_sf_bytes(rows, kb))


def mx_sf_bytes_x4(rows: int, kb: int) -> int:
    return int(load().mx_sf_bytes_x4(rows, kb))


def mx_padded_rows_bound(R: int, E: int) -> int:
    return int(load().mx_padded_rows_bound(R, E))


def moe_permute_workspace_bytes(T: int, k: int, E: int) -> int:
    return int(load().moe_permute_workspace_bytes(T, k, E))


# ------------------------------------------------------------------ raw calls
def mxfp8_quantize(x, rows, cols, mode, seg_off, seg_poff, nseg, ld_col, q_row, sf_row, q_col, sf_col,
                   dev_err=None, stream=None):
    st = load().mxfp8_quantize(_ptr(x), rows, cols, mode, _ptr(seg_off), _ptr(seg_poff), nseg, ld_col, _ptr(q_row),
                               _ptr(sf_row), _ptr(q_col), _ptr(sf_col), _ptr(dev_err), _stream(stream))
    _check(st, "mxfp8_quantize")


def mxfp8_quantize_ex(x, dtype, scale_rule, rows, cols, mode, seg_off, seg_poff, nseg, ld_col, q_row, sf_row,
                      q_col, sf_col, dev_err=None, stream=None):
    st = load().mxfp8_quantize_ex(_ptr(x), dtype, scale_rule, rows, cols, mode, _ptr(seg_off), _ptr(seg_poff), nseg,
                                  ld_col, _ptr(q_row), _ptr(sf_row), _ptr(q_col), _ptr(sf_col), _ptr(dev_err),
                                  _stream(stream))
    _check(st, "mxfp8_quantize_ex")


def mxfp8_swiglu_quantize(a, R, I, mode, seg_off, seg_poff, nseg, ld_col, q_row, sf_row, q_col, sf_col,
                          dev_err=None, stream=None):
    st = load().mxfp8_swiglu_quantize(_ptr(a), R, I, mode, _ptr(seg_off), _ptr(seg_poff), nseg, ld_col, _ptr(q_row),
                                      _ptr(sf_row), _ptr(q_col), _ptr(sf_col), _ptr(dev_err), _stream(stream))
    _check(st, "mxfp8_swiglu_quantize")


def mxfp8_swiglu_bwd_quantize(dh, a, R, I, mode, seg_off, seg_poff, nseg, ld_col, q_row, sf_row, q_col, sf_col,
                              dev_err=None, stream=None):
    st = load().mxfp8_swiglu_bwd_quantize(_ptr(dh), _ptr(a), R, I, mode, _ptr(seg_off), _ptr(seg_poff), nseg,
                                          ld_col, _ptr(q_row), _ptr(sf_row), _ptr(q_col), _ptr(sf_col),
                                          _ptr(dev_err), _stream(stream))
    _check(st, "mxfp8_swiglu_bwd_quantize")


def mxfp8_gather_quantize(x, T, cols, mode, src_row, off, poff, E, R, ld_col, q_row, sf_row, q_col, sf_col,
                          dev_err, stream=None):
    st = load().mxfp8_gather_quantize(_ptr(x), T, cols, mode, _ptr(src_row), _ptr(off), _ptr(poff), E, R, ld_col,
                                      _ptr(q_row), _ptr(sf_row), _ptr(q_col), _ptr(sf_col), _ptr(dev_err),
                                      _stream(stream))
    _check(st, "mxfp8_gather_quantize")


def mxfp8_gather_quantize_ex(x, T, cols, mode, src_row, row_scale, off, poff, E, R, ld_col, q_row, sf_row, q_col,
                             sf_col, dev_err, stream=None):
    st = load().mxfp8_gather_quantize_ex(_ptr(x), T, cols, mode, _ptr(src_row), _ptr(row_scale), _ptr(off),
                                         _ptr(poff), E, R, ld_col, _ptr(q_row), _ptr(sf_row), _ptr(q_col),
                                         _ptr(sf_col), _ptr(dev_err), _stream(stream))
    _check(st, "mxfp8_gather_quantize_ex")


def moe_permute(topk_ids, T, k, E, counts, off, poff, src_row, dst_of, q_in, sf_in, K, q_out, sf_out, ws,
                ws_bytes, dev_err, stream=None):
    st = load().moe_permute(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(off), _ptr(poff), _ptr(src_row),
                            _ptr(dst_of), _ptr(q_in), _ptr(sf_in), K, _ptr(q_out), _ptr(sf_out), _ptr(ws),
                            ws_bytes, _ptr(dev_err), _stream(stream))
    _check(st, "moe_permute")


def moe_permute_noalloc(topk_ids, T, k, E, counts, off, poff, src_row, dst_of, q_in, sf_in, K, q_out, sf_out,
                        dev_err, stream=None):
    """moe_permute with the library's fixed device scratch instead of a caller workspace."""
    st = load().moe_permute_noalloc(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(off), _ptr(poff), _ptr(src_row),
                                    _ptr(dst_of), _ptr(q_in), _ptr(sf_in), K, _ptr(q_out), _ptr(sf_out),
                                    _ptr(dev_err), _stream(stream))
    _check(st, "moe_permute_noalloc")


def moe_gather_rows(src, row_bytes, src_row, R, dst, stream=None):
    st = load().moe_gather_rows(_ptr(src), row_bytes, _ptr(src_row), R, _ptr(dst), _stream(stream))
    _check(st, "moe_gather_rows")


def moe_combine_fwd(Y, gate, dst_of, T, k, H, R, out, dev_err, stream=None):
    st = load().moe_combine_fwd(_ptr(Y), _ptr(gate), _ptr(dst_of), T, k, H, R, _ptr(out), _ptr(dev_err),
                                _stream(stream))
    _check(st, "moe_combine_fwd")


def moe_combine_bwd(dOut, Y, gate, dst_of, T, k, H, R, dY, dgate, dev_err, stream=None):
    st = load().moe_combine_bwd(_ptr(dOut), _ptr(Y), _ptr(gate), _ptr(dst_of), T, k, H, R, _ptr(dY), _ptr(dgate),
                                _ptr(dev_err), _stream(stream))
    _check(st, "moe_combine_bwd")


def moe_combine_bwd_ex(dOut, Y, gate, dst_of, T, k, H, R, dY, dgate, gate_rows, dev_err, stream=None):
    st = load().moe_combine_bwd_ex(_ptr(dOut), _ptr(Y), _ptr(gate), _ptr(dst_of), T, k, H, R, _ptr(dY), _ptr(dgate),
                                   _ptr(gate_rows), _ptr(dev_err), _stream(stream))
    _check(st, "moe_combine_bwd_ex")


def grouped_gemm_mxfp8_fwd(A, SFA, B, SFB, off, poff, E, R, N, K, C, dev_err, stream=None):
    st = load().grouped_gemm_mxfp8_fwd(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(off), _ptr(poff), E, R, N, K,
                                       _ptr(C), _ptr(dev_err), _stream(stream))
    _check(st, "grouped_gemm_mxfp8_fwd")


def grouped_gemm_mxfp8_fwd_swiglu(A, SFA, W1, SFW1, off, poff, E, R, I, K, out1, h_qrow, h_sfrow, h_qcol, h_sfcol,
                                  ld_col, h_mode, dev_err, stream=None):
    st = load().grouped_gemm_mxfp8_fwd_swiglu(_ptr(A), _ptr(SFA), _ptr(W1), _ptr(SFW1), _ptr(off), _ptr(poff), E, R, I,
                                              K, _ptr(out1), _ptr(h_qrow), _ptr(h_sfrow), _ptr(h_qcol), _ptr(h_sfcol),
                                              ld_col, h_mode, _ptr(dev_err), _stream(stream))
    _check(st, "grouped_gemm_mxfp8_fwd_swiglu")


def grouped_gemm_mxfp8_dgrad(dY, SFdY, Wt, SFWt, off, poff, E, R, N, K, dX, dev_err, stream=None):
    st = load().grouped_gemm_mxfp8_dgrad(_ptr(dY), _ptr(SFdY), _ptr(Wt), _ptr(SFWt), _ptr(off), _ptr(poff), E, R, N,
                                         K, _ptr(dX), _ptr(dev_err), _stream(stream))
    _check(st, "grouped_gemm_mxfp8_dgrad")


def grouped_gemm_mxfp8_wgrad(dYc, SFdYc, Xc, SFXc, off, poff, E, N, K, ld_tok, dW, dev_err, stream=None):
    st = load().grouped_gemm_mxfp8_wgrad(_ptr(dYc), _ptr(SFdYc), _ptr(Xc), _ptr(SFXc), _ptr(off), _ptr(poff), E, N,
                                         K, ld_tok, _ptr(dW), _ptr(dev_err), _stream(stream))
    _check(st, "grouped_gemm_mxfp8_wgrad")


def grouped_gemm_mxfp8_fwd_ex(A, SFA, B, SFB, off, poff, E, R, N, K, C, flags, dev_err, stream=None):
    st = load().grouped_gemm_mxfp8_fwd_ex(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(off), _ptr(poff), E, R, N, K,
                                          _ptr(C), flags, _ptr(dev_err), _stream(stream))
    _check(st, "grouped_gemm_mxfp8_fwd_ex")


def grouped_gemm_mxfp8_fwd_swiglu_ex(A, SFA, W1, SFW1, off, poff, E, R, I, K, out1, h_qrow, h_sfrow, h_qcol, h_sfcol,
                                     ld_col, h_mode, flags, dev_err, stream=None):
    st = load().grouped_gemm_mxfp8_fwd_swiglu_ex(_ptr(A), _ptr(SFA), _ptr(W1), _ptr(SFW1), _ptr(off), _ptr(poff), E,
                                                 R, I, K, _ptr(out1), _ptr(h_qrow), _ptr(h_sfrow), _ptr(h_qcol),
                                                 _ptr(h_sfcol), ld_col, h_mode, flags, _ptr(dev_err), _stream(stream))
    _check(st, "grouped_gemm_mxfp8_fwd_swiglu_ex")


def grouped_gemm_mxfp8_dgrad_ex(dY, SFdY, Wt, SFWt, off, poff, E, R, N, K, dX, flags, dev_err, stream=None):
    st = load().grouped_gemm_mxfp8_dgrad_ex(_ptr(dY), _ptr(SFdY), _ptr(Wt), _ptr(SFWt), _ptr(off), _ptr(poff), E, R,
                                            N, K, _ptr(dX), flags, _ptr(dev_err), _stream(stream))
    _check(st, "grouped_gemm_mxfp8_dgrad_ex")


def grouped_gemm_mxfp8_wgrad_ex(dYc, SFdYc, Xc, SFXc, off, poff, E, N, K, ld_tok, dW, flags, dev_err, stream=None):
    st = load().grouped_gemm_mxfp8_wgrad_ex(_ptr(dYc), _ptr(SFdYc), _ptr(Xc), _ptr(SFXc), _ptr(off), _ptr(poff), E,
                                            N, K, ld_tok, _ptr(dW), flags, _ptr(dev_err), _stream(stream))
    _check(st, "grouped_gemm_mxfp8_wgrad_ex")


def testing_grouped_gemm(pass_, A, SFA, B, SFB, off, poff, E, R, N, K, ld_tok, out, dev_err, flags=0,
                         ctas_per_mma=0, wait_limit_ns=0, withhold_operands=False, raster_group=0,
                         cluster_pairs=0, stream=None) -> int:
    """mx_testing_grouped_gemm (tests and A/B measurements only); returns the status code."""
    opt = TestingGemmOptions(ctas_per_mma, wait_limit_ns, 1 if withhold_operands else 0, raster_group,
                             cluster_pairs)
    return int(load().mx_testing_grouped_gemm(pass_, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(off), _ptr(poff), E,
                                              R, N, K, ld_tok, _ptr(out), flags, ctypes.byref(opt), _ptr(dev_err),
                                              _stream(stream)))


# ------------------------------------------------------------------ allocating helpers
def new_dev_err(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)


def quantize_alloc(x: torch.Tensor, mode: int = MX_ROWWISE, seg_off=None, seg_poff=None, dev_err=None,
                   stream=None, ld_col=None, scale_rule: int = MX_SCALE_FLOOR) -> dict:
    """Quantize a bf16 [rows, cols] CUDA tensor; returns the output tensors in a dict.

    ld_col defaults to the padded-position bound; pass it explicitly when the
    segments are known to need less (e.g. weights stacked with 128-multiple rows)."""
    assert x.dtype in (torch.bfloat16, torch.float32) and x.dim() == 2
    rows, cols = x.shape
    nseg = 0 if seg_off is None else seg_off.numel() - 1
    pbound = mx_padded_rows_bound(rows, nseg) if nseg else (rows + 127) // 128 * 128
    if ld_col is None:
        ld_col = pbound
    dev = x.device
    out = dict(pbound=pbound, ld_col=ld_col)
    q_row = sf_row = q_col = sf_col = None
    if mode & MX_ROWWISE:
        q_row = torch.empty(rows, cols, dtype=torch.uint8, device=dev)
        nb = (mx_sf_bytes_x4 if mode & MX_ROWWISE_X4 else mx_sf_bytes)(pbound, cols // 32)
        sf_row = torch.empty(nb, dtype=torch.uint8, device=dev)
    if mode & MX_COLWISE:
        q_col = torch.empty(cols, ld_col, dtype=torch.uint8, device=dev)
        nb = (mx_sf_bytes_x4 if mode & MX_COLWISE_X4 else mx_sf_bytes)(cols, ld_col // 32)
        sf_col = torch.empty(nb, dtype=torch.uint8, device=dev)
    dtype = MX_DTYPE_F32 if x.dtype == torch.float32 else MX_DTYPE_BF16
    mxfp8_quantize_ex(x, dtype, scale_rule, rows, cols, mode, seg_off, seg_poff, nseg, ld_col, q_row, sf_row, q_col,
                      sf_col, dev_err, stream)
    out.update(q_row=q_row, sf_row=sf_row, q_col=q_col, sf_col=sf_col)
    return out


def permute_alloc(topk_ids: torch.Tensor, E: int, q_in=None, sf_in=None, dev_err=None, stream=None) -> dict:
    T, k = topk_ids.shape
    dev = topk_ids.device
    R = T * k
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
               off=torch.empty(E + 1, dtype=torch.int32, device=dev),
               poff=torch.empty(E + 1, dtype=torch.int32, device=dev),
               src_row=torch.empty(max(R, 1), dtype=torch.int32, device=dev),
               dst_of=torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    wsb = moe_permute_workspace_bytes(T, k, E)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    if dev_err is None:
        dev_err = new_dev_err(dev)
    K = 0
    q_out = sf_out = None
    if q_in is not None:
        K = q_in.shape[1]
        q_out = torch.empty(max(R, 1), K, dtype=torch.uint8, device=dev)
        sf_out = torch.empty(mx_sf_bytes(mx_padded_rows_bound(R, E), K // 32), dtype=torch.uint8, device=dev)
    moe_permute(topk_ids, T, k, E, out["counts"], out["off"], out["poff"], out["src_row"], out["dst_of"], q_in,
                sf_in, K, q_out, sf_out, ws, wsb, dev_err, stream)
    out.update(q=q_out, sf=sf_out, dev_err=dev_err, ws=ws)
    return out
