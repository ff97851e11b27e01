"""ctypes binding of libnvfp4moe.so: one Python function per C entry point,
with the same name and parameter order.  Tensors stand in for pointers
(``None`` for NULL); every step of the path runs in the library's kernels.
A non-zero status raises ``NvError``.  Nothing here computes on the CPU, and a
missing library raises instead of falling back.

Allocation helpers (``*_sizes``) only report buffer shapes from the library's
own size functions.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libnvfp4moe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "nvfp4moe.h")

NV_OK, NV_ERR_ARG, NV_ERR_ALIGN, NV_ERR_SHAPE, NV_ERR_OFFSETS = 0, -1, -2, -3, -4
NV_ERR_TIMEOUT, NV_ERR_CUDA, NV_ERR_UNSUPPORTED, NV_ERR_WORKSPACE = -5, -6, -7, -8
NV_RN, NV_SR = 0, 1
NV_OUT_BF16, NV_OUT_FP32 = 0, 1

_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_U64 = ctypes.c_uint64
_SZ = ctypes.c_size_t

_SIGS = {
    "nvfp4moe_padded_cap": (_I64, [_I64, _I64]),
    "nvfp4moe_scale_bytes": (_I64, [_I64, _I64]),
    "nvfp4moe_scale_offset": (_I64, [_I64, _I64, _I64]),
    "nvfp4moe_quantize_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "nvfp4moe_quantize_gather_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "nvfp4moe_fwd_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "nvfp4_quantize": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_quantize_noalloc": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P]),
    "nvfp4_quantize_requant": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P, _SZ, _U64, _U64,
                                              _P, _P, _P]),
    "mxfp8_quantize": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, ctypes.c_int, _U64, _U64, _U64,
                                      _P, _P, _P, _P, _P]),
    "dequant_transpose_requant_sr": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P, _I32, _U64, _U64,
                                                    _P, _P, _P]),
    "grouped_gemm_nvfp4_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64,
                                              _P, ctypes.c_int, _P, _SZ, _P]),
    "grouped_gemm_nvfp4_fwd_swiglu": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _P, _P,
                                                     _P, _P]),
    "grouped_gemm_mxfp8_dx": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _P, ctypes.c_int,
                                             _P, _SZ, _P]),
    "grouped_gemm_mxfp8_dx_swiglu_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _P, _P, _P]),
    "grouped_gemm_mxfp8_dw": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _P, _P, _SZ, _P]),
    "rht32_s2f6_quantize": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_uint32, _P, _P, _P]),
    "s2f6_dequantize_rht32_inverse": (ctypes.c_int, [_P, _P, _I64, _I64, ctypes.c_uint32, _P, ctypes.c_int, _P]),
    "nvfp4moe_swiglu_fwd": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "nvfp4moe_swiglu_bwd": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
    "nvfp4moe_get_device_status": (ctypes.c_int, [_P]),
    "nvfp4moe_selftest_wait_timeout": (ctypes.c_int, [_I64, _P]),
    "nvfp4moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "nvfp4moe_version": (ctypes.c_char_p, []),
    "nvfp4moe_set_gemm_kernel": (ctypes.c_int, [ctypes.c_int]),
    "nvfp4moe_set_gemm_wait_limit": (ctypes.c_int, [_I64]),
    "nvfp4moe_sr_e4m3x4": (ctypes.c_int, [_P, _P, _I64, _P, _P]),
    "nvfp4_quantize_requant_gather": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P, _SZ,
                                                     _U64, _U64, _P, _P, _P]),
    "grouped_gemm_nvfp4_fwd_rht_s2f6": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64,
                                                       ctypes.c_uint32, _P, _P, _P, _P]),
    "nvfp4_outer_scale": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _SZ, _P]),
    "nvfp4_quantize_four_over_six": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_quantize_requant_four_over_six": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P, _SZ,
                                                            _U64, _U64, _P, _P, _P]),
    "nvfp4_quantize_rows": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P]),
    "nvfp4_quantize_requant_rows": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _P, _P, _P, _P, _U64, _U64, _P, _P,
                                                   _P]),
    "dequant_transpose_requant_sr_rows": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _P, _I32, _U64, _U64, _P, _P,
                                                         _P]),
    "grouped_gemm_nvfp4_fwd_rows": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _P,
                                                   ctypes.c_int, _P]),
    "grouped_gemm_nvfp4_fwd_swiglu_rows": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _P,
                                                          _P, _P, _P]),
}


class NvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({status_string(status)})")
        self.status = status


def lib():
    """The loaded library.  Raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m precision_moe_numerics_nvfp4_gb300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def declared_functions():
    """Names of the functions include/nvfp4moe.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", txt, flags=re.M))
                  - {"if", "while", "for", "return", "sizeof"})


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if not t.is_cuda:
        raise ValueError("device tensors only")
    if not t.is_contiguous():
        raise ValueError("contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(name, status):
    if status != NV_OK:
        raise NvError(name, status)
    return status


def _ng(group_offsets):
    return 0 if group_offsets is None else group_offsets.numel() - 1


# ---- host helpers -------------------------------------------------------------
def nvfp4moe_padded_cap(M_total: int, E: int) -> int:
    return int(lib().nvfp4moe_padded_cap(M_total, E))


def nvfp4moe_scale_bytes(padded_rows: int, kblocks: int) -> int:
    return int(lib().nvfp4moe_scale_bytes(padded_rows, kblocks))


def nvfp4moe_scale_offset(rp: int, c: int, kblocks: int) -> int:
    return int(lib().nvfp4moe_scale_offset(rp, c, kblocks))


def nvfp4moe_quantize_workspace_bytes(batch: int, rows: int, cols: int) -> int:
    return int(lib().nvfp4moe_quantize_workspace_bytes(batch, rows, cols))


def nvfp4moe_quantize_gather_workspace_bytes(src_rows: int, rows: int, cols: int) -> int:
    return int(lib().nvfp4moe_quantize_gather_workspace_bytes(src_rows, rows, cols))


def nvfp4moe_fwd_workspace_bytes(M_total: int, K: int, E: int) -> int:
    return int(lib().nvfp4moe_fwd_workspace_bytes(M_total, K, E))


def status_string(status: int) -> str:
    return lib().nvfp4moe_status_string(status).decode()


def nvfp4moe_version() -> str:
    return lib().nvfp4moe_version().decode()


GEMM_AUTO, GEMM_ONE_PER_SM, GEMM_TWO_PER_SM, GEMM_CTA_PAIR, GEMM_CTA_PAIR_N128 = 0, 1, 2, 3, 4


def nvfp4moe_set_gemm_kernel(variant: int) -> None:
    """Kernel choice of the grouped GEMMs: GEMM_AUTO, GEMM_ONE_PER_SM,
    GEMM_TWO_PER_SM, GEMM_CTA_PAIR (256 x 256 pair tiles) or
    GEMM_CTA_PAIR_N128 (256 x 128 pair tiles, two pairs per SM pair); a pair
    choice applies where the shape allows it."""
    _check("nvfp4moe_set_gemm_kernel", lib().nvfp4moe_set_gemm_kernel(int(variant)))


def nvfp4_quantize_requant_gather(x, row_src, src_rows, rows, cols, group_offsets, outer_scale_in, outer_scale_out,
                                  codes, scales, workspace, seed, counter_offset, out_codes, out_scales, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("nvfp4_quantize_requant_gather", lib().nvfp4_quantize_requant_gather(
        _ptr(x), _ptr(row_src), int(src_rows), int(rows), int(cols), _ptr(group_offsets), _ng(group_offsets),
        _ptr(outer_scale_in), _ptr(outer_scale_out), _ptr(codes), _ptr(scales), _ptr(workspace), ws_bytes, seed,
        counter_offset, _ptr(out_codes), _ptr(out_scales), _stream(stream)))


def nvfp4moe_sr_e4m3x4(x, draws, n4, codes, stream=None):
    """codes[4i + k] = the library's SR of x[4i + k] to E4M3 with the draws
    draws[i] = U_a | U_b << 16 (see the header)."""
    return _check("nvfp4moe_sr_e4m3x4", lib().nvfp4moe_sr_e4m3x4(_ptr(x), _ptr(draws), int(n4), _ptr(codes),
                                                                  _stream(stream)))


def nvfp4moe_set_gemm_wait_limit(spins: int) -> None:
    """Iteration limit of the grouped GEMMs' pipeline waits (0: the default);
    a tiny limit makes them run out (a test of the bounded-wait path)."""
    _check("nvfp4moe_set_gemm_wait_limit", lib().nvfp4moe_set_gemm_wait_limit(int(spins)))


# ---- the hot path -------------------------------------------------------------
def nvfp4_quantize(x, batch, rows, cols, group_offsets, outer_scale_in, outer_scale_out, codes, scales,
                   workspace, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("nvfp4_quantize", lib().nvfp4_quantize(
        _ptr(x), batch, rows, cols, _ptr(group_offsets), _ng(group_offsets), _ptr(outer_scale_in),
        _ptr(outer_scale_out), _ptr(codes), _ptr(scales), _ptr(workspace), ws_bytes, _stream(stream)))


def nvfp4_quantize_noalloc(x, batch, rows, cols, group_offsets, outer_scale_in, outer_scale_out, codes, scales,
                           stream=None):
    """nvfp4_quantize without a workspace argument, for callers that cannot
    allocate device memory: the library uses its own fixed scratch."""
    return _check("nvfp4_quantize_noalloc", lib().nvfp4_quantize_noalloc(
        _ptr(x), batch, rows, cols, _ptr(group_offsets), _ng(group_offsets), _ptr(outer_scale_in),
        _ptr(outer_scale_out), _ptr(codes), _ptr(scales), _stream(stream)))


def nvfp4_quantize_requant(x, batch, rows, cols, group_offsets, outer_scale_in, outer_scale_out, codes, scales,
                           workspace, seed, counter_offset, out_codes, out_scales, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("nvfp4_quantize_requant", lib().nvfp4_quantize_requant(
        _ptr(x), batch, rows, cols, _ptr(group_offsets), _ng(group_offsets), _ptr(outer_scale_in),
        _ptr(outer_scale_out), _ptr(codes), _ptr(scales), _ptr(workspace), ws_bytes, seed, counter_offset,
        _ptr(out_codes), _ptr(out_scales), _stream(stream)))


def mxfp8_quantize(x, rows, cols, group_offsets, mode, seed, counter_offset_row, counter_offset_t,
                   codes_row, scales_row, codes_t, scales_t, stream=None):
    return _check("mxfp8_quantize", lib().mxfp8_quantize(
        _ptr(x), rows, cols, _ptr(group_offsets), _ng(group_offsets), mode, seed, counter_offset_row,
        counter_offset_t, _ptr(codes_row), _ptr(scales_row), _ptr(codes_t), _ptr(scales_t), _stream(stream)))


def dequant_transpose_requant_sr(codes, scales, outer_scale, batch, rows, cols, group_offsets, seed,
                                 counter_offset, out_codes, out_scales, stream=None):
    return _check("dequant_transpose_requant_sr", lib().dequant_transpose_requant_sr(
        _ptr(codes), _ptr(scales), _ptr(outer_scale), batch, rows, cols, _ptr(group_offsets), _ng(group_offsets),
        seed, counter_offset, _ptr(out_codes), _ptr(out_scales), _stream(stream)))


def grouped_gemm_nvfp4_fwd(x_bf16, x_outer_scale, x_codes, x_scales, w_codes, w_scales, w_outer_scale,
                           group_offsets, E, M_total, N, K, y, y_dtype, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("grouped_gemm_nvfp4_fwd", lib().grouped_gemm_nvfp4_fwd(
        _ptr(x_bf16), _ptr(x_outer_scale), _ptr(x_codes), _ptr(x_scales), _ptr(w_codes), _ptr(w_scales),
        _ptr(w_outer_scale), _ptr(group_offsets), E, M_total, N, K, _ptr(y), y_dtype, _ptr(workspace), ws_bytes,
        _stream(stream)))


def rht32_s2f6_quantize(x, rows, cols, signs, codes, scales, stream=None):
    return _check("rht32_s2f6_quantize", lib().rht32_s2f6_quantize(
        _ptr(x), rows, cols, int(signs) & 0xFFFFFFFF, _ptr(codes), _ptr(scales), _stream(stream)))


def s2f6_dequantize_rht32_inverse(codes, scales, rows, cols, signs, y, y_dtype, stream=None):
    return _check("s2f6_dequantize_rht32_inverse", lib().s2f6_dequantize_rht32_inverse(
        _ptr(codes), _ptr(scales), rows, cols, int(signs) & 0xFFFFFFFF, _ptr(y), y_dtype, _stream(stream)))


def grouped_gemm_nvfp4_fwd_swiglu(x_outer_scale, x_codes, x_scales, w13_codes, w13_scales, w13_outer_scale,
                                  group_offsets, E, M_total, I, K, y13, h, h_outer_scale, stream=None):
    return _check("grouped_gemm_nvfp4_fwd_swiglu", lib().grouped_gemm_nvfp4_fwd_swiglu(
        _ptr(x_outer_scale), _ptr(x_codes), _ptr(x_scales), _ptr(w13_codes), _ptr(w13_scales),
        _ptr(w13_outer_scale), _ptr(group_offsets), E, M_total, I, K, _ptr(y13), _ptr(h), _ptr(h_outer_scale),
        _stream(stream)))


def nvfp4_outer_scale(x, batch, n, outer_scale_out, workspace, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("nvfp4_outer_scale", lib().nvfp4_outer_scale(
        _ptr(x), batch, n, _ptr(outer_scale_out), _ptr(workspace), ws_bytes, _stream(stream)))


def nvfp4_quantize_four_over_six(x, batch, rows, cols, group_offsets, outer_scale_in, outer_scale_out, codes, scales,
                                 workspace, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("nvfp4_quantize_four_over_six", lib().nvfp4_quantize_four_over_six(
        _ptr(x), batch, rows, cols, _ptr(group_offsets), _ng(group_offsets), _ptr(outer_scale_in),
        _ptr(outer_scale_out), _ptr(codes), _ptr(scales), _ptr(workspace), ws_bytes, _stream(stream)))


def nvfp4_quantize_requant_four_over_six(x, batch, rows, cols, group_offsets, outer_scale_in, outer_scale_out, codes,
                                         scales, workspace, seed, counter_offset, out_codes, out_scales, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("nvfp4_quantize_requant_four_over_six", lib().nvfp4_quantize_requant_four_over_six(
        _ptr(x), batch, rows, cols, _ptr(group_offsets), _ng(group_offsets), _ptr(outer_scale_in),
        _ptr(outer_scale_out), _ptr(codes), _ptr(scales), _ptr(workspace), ws_bytes, seed, counter_offset,
        _ptr(out_codes), _ptr(out_scales), _stream(stream)))


def grouped_gemm_nvfp4_fwd_rht_s2f6(x_outer_scale, x_codes, x_scales, w_codes, w_scales, w_outer_scale,
                                    group_offsets, E, M_total, N, K, signs, y, codes, scales, stream=None):
    return _check("grouped_gemm_nvfp4_fwd_rht_s2f6", lib().grouped_gemm_nvfp4_fwd_rht_s2f6(
        _ptr(x_outer_scale), _ptr(x_codes), _ptr(x_scales), _ptr(w_codes), _ptr(w_scales), _ptr(w_outer_scale),
        _ptr(group_offsets), E, M_total, N, K, int(signs) & 0xFFFFFFFF, _ptr(y), _ptr(codes), _ptr(scales),
        _stream(stream)))


# ---- per-token activation outer scales ------------------------------------------------
def nvfp4_quantize_rows(x, rows, cols, group_offsets, sg_rows_in, sg_rows_out, codes, scales, stream=None):
    return _check("nvfp4_quantize_rows", lib().nvfp4_quantize_rows(
        _ptr(x), rows, cols, _ptr(group_offsets), _ng(group_offsets), _ptr(sg_rows_in), _ptr(sg_rows_out),
        _ptr(codes), _ptr(scales), _stream(stream)))


def nvfp4_quantize_requant_rows(x, rows, cols, group_offsets, sg_rows_in, sg_rows_out, codes, scales, seed,
                                counter_offset, out_codes, out_scales, stream=None):
    return _check("nvfp4_quantize_requant_rows", lib().nvfp4_quantize_requant_rows(
        _ptr(x), rows, cols, _ptr(group_offsets), _ng(group_offsets), _ptr(sg_rows_in), _ptr(sg_rows_out),
        _ptr(codes), _ptr(scales), seed, counter_offset, _ptr(out_codes), _ptr(out_scales), _stream(stream)))


def dequant_transpose_requant_sr_rows(codes, scales, sg_rows, rows, cols, group_offsets, seed, counter_offset,
                                      out_codes, out_scales, stream=None):
    return _check("dequant_transpose_requant_sr_rows", lib().dequant_transpose_requant_sr_rows(
        _ptr(codes), _ptr(scales), _ptr(sg_rows), rows, cols, _ptr(group_offsets), _ng(group_offsets), seed,
        counter_offset, _ptr(out_codes), _ptr(out_scales), _stream(stream)))


def grouped_gemm_nvfp4_fwd_rows(x_sg_rows, x_codes, x_scales, w_codes, w_scales, w_outer_scale, group_offsets, E,
                                M_total, N, K, y, y_dtype, stream=None):
    return _check("grouped_gemm_nvfp4_fwd_rows", lib().grouped_gemm_nvfp4_fwd_rows(
        _ptr(x_sg_rows), _ptr(x_codes), _ptr(x_scales), _ptr(w_codes), _ptr(w_scales), _ptr(w_outer_scale),
        _ptr(group_offsets), E, M_total, N, K, _ptr(y), y_dtype, _stream(stream)))


def grouped_gemm_nvfp4_fwd_swiglu_rows(x_sg_rows, x_codes, x_scales, w13_codes, w13_scales, w13_outer_scale,
                                       group_offsets, E, M_total, I, K, y13, h, h_sg_rows, stream=None):
    return _check("grouped_gemm_nvfp4_fwd_swiglu_rows", lib().grouped_gemm_nvfp4_fwd_swiglu_rows(
        _ptr(x_sg_rows), _ptr(x_codes), _ptr(x_scales), _ptr(w13_codes), _ptr(w13_scales), _ptr(w13_outer_scale),
        _ptr(group_offsets), E, M_total, I, K, _ptr(y13), _ptr(h), _ptr(h_sg_rows), _stream(stream)))


def grouped_gemm_mxfp8_dx(g_codes, g_scales, wt_codes, wt_scales, group_offsets, E, M_total, N, K, dx, dx_dtype,
                          workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("grouped_gemm_mxfp8_dx", lib().grouped_gemm_mxfp8_dx(
        _ptr(g_codes), _ptr(g_scales), _ptr(wt_codes), _ptr(wt_scales), _ptr(group_offsets), E, M_total, N, K,
        _ptr(dx), dx_dtype, _ptr(workspace), ws_bytes, _stream(stream)))


def grouped_gemm_mxfp8_dx_swiglu_bwd(g_codes, g_scales, wt_codes, wt_scales, group_offsets, E, M_total, N, I, y13,
                                     dy13, stream=None):
    return _check("grouped_gemm_mxfp8_dx_swiglu_bwd", lib().grouped_gemm_mxfp8_dx_swiglu_bwd(
        _ptr(g_codes), _ptr(g_scales), _ptr(wt_codes), _ptr(wt_scales), _ptr(group_offsets), E, M_total, N, I,
        _ptr(y13), _ptr(dy13), _stream(stream)))


def grouped_gemm_mxfp8_dw(gt_codes, gt_scales, xt_codes, xt_scales, group_offsets, E, M_total, N, K, dw,
                          workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check("grouped_gemm_mxfp8_dw", lib().grouped_gemm_mxfp8_dw(
        _ptr(gt_codes), _ptr(gt_scales), _ptr(xt_codes), _ptr(xt_scales), _ptr(group_offsets), E, M_total, N, K,
        _ptr(dw), _ptr(workspace), ws_bytes, _stream(stream)))


def nvfp4moe_swiglu_fwd(y13, M, I, h, stream=None):
    return _check("nvfp4moe_swiglu_fwd", lib().nvfp4moe_swiglu_fwd(_ptr(y13), M, I, _ptr(h), _stream(stream)))


def nvfp4moe_swiglu_bwd(dh, y13, M, I, dy13, stream=None):
    return _check("nvfp4moe_swiglu_bwd", lib().nvfp4moe_swiglu_bwd(_ptr(dh), _ptr(y13), M, I, _ptr(dy13),
                                                                   _stream(stream)))


def nvfp4moe_get_device_status(stream=None) -> int:
    """Status word of the current device (synchronizes the stream); clears it."""
    return int(lib().nvfp4moe_get_device_status(_stream(stream)))


def nvfp4moe_selftest_wait_timeout(spins: int, stream=None):
    return _check("nvfp4moe_selftest_wait_timeout", lib().nvfp4moe_selftest_wait_timeout(spins, _stream(stream)))


# ---- buffer shapes ---------------------------------------------------------------
def nvfp4_sizes(batch: int, rows: int, cols: int, E: int | None = None):
    """(codes bytes, scale bytes) of nvfp4_quantize; E selects the grouped layout."""
    if E is None:
        prow = batch * ((rows + 127) // 128 * 128)
    else:
        prow = nvfp4moe_padded_cap(rows, E)
    return batch * rows * (cols // 2), nvfp4moe_scale_bytes(prow, cols // 16)


def mxfp8_row_sizes(rows: int, cols: int, E: int | None = None):
    prow = nvfp4moe_padded_cap(rows, E) if E else (rows + 127) // 128 * 128
    return rows * cols, nvfp4moe_scale_bytes(prow, cols // 32)


def mxfp8_t_sizes(rows: int, cols: int, E: int | None = None):
    """(P_cap, codes bytes, scale bytes) of a transposed-per-group output."""
    P = nvfp4moe_padded_cap(rows, E) if E else (rows + 127) // 128 * 128
    return P, cols * P, nvfp4moe_scale_bytes(cols, P // 32)


def requant_weight_sizes(batch: int, rows: int, cols: int):
    """(codes bytes, scale bytes) of dequant_transpose_requant_sr on weights."""
    cpad = (cols + 127) // 128 * 128
    return batch * cols * rows, nvfp4moe_scale_bytes(batch * cpad, rows // 32)
