"""Argument validation of the C-ABI entry points, on the host: every call
checks its pointers, sizes, shape rules and alignment before touching the
GPU, so these run without one.  The addresses are never dereferenced (each
case fails validation, or is an empty problem that returns at once)."""
import ctypes

import pytest

from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N

A = ctypes.c_void_p(1 << 24)            # 32-byte aligned fake device address
A16 = ctypes.c_void_p((1 << 24) + 16)   # 16- but not 32-byte aligned
A4 = ctypes.c_void_p((1 << 24) + 4)     # 4- but not 16-byte aligned
A1 = ctypes.c_void_p((1 << 24) + 1)     # byte aligned only
NULL = None
S = None                                # default stream


@pytest.fixture(scope="module")
def L():
    from precision_moe_numerics_nvfp4_gb300 import build
    build.build()
    return N.lib()


def test_quantize_rows_validation(L):
    f = L.nvfp4_quantize_rows
    assert f(NULL, 128, 128, NULL, 0, NULL, A, A, A, S) == N.NV_ERR_ARG           # no x
    assert f(A, 128, 128, NULL, 0, NULL, NULL, A, A, S) == N.NV_ERR_ARG           # no scale in or out
    assert f(A, 128, 120, NULL, 0, NULL, A, A, A, S) == N.NV_ERR_SHAPE            # cols % 16
    assert f(A4, 128, 128, NULL, 0, NULL, A, A, A, S) == N.NV_ERR_ALIGN           # x not 16-byte aligned
    assert f(A, 128, 128, NULL, 0, NULL, A1, A, A, S) == N.NV_ERR_ALIGN           # row scales not 4-byte aligned
    assert f(A, 128, 128, A, 0, NULL, A, A, A, S) == N.NV_ERR_ARG                 # groups without a count
    assert f(A, 0, 128, NULL, 0, NULL, A, A, A, S) == N.NV_OK                     # empty: nothing launched
    g = L.nvfp4_quantize_requant_rows
    assert g(A, 128, 192, NULL, 0, NULL, A, A, A, 1, 0, A, A, S) == N.NV_ERR_SHAPE   # cols % 128
    assert g(A, 100, 128, NULL, 0, NULL, A, A, A, 1, 0, A, A, S) == N.NV_ERR_SHAPE   # plain rows % 128
    assert g(A, 128, 128, NULL, 0, NULL, A, A, A, 1, 0, NULL, A, S) == N.NV_ERR_ARG
    h = L.dequant_transpose_requant_sr_rows
    assert h(A, A, NULL, 128, 128, NULL, 0, 1, 0, A, A, S) == N.NV_ERR_ARG         # no row scales
    assert h(A, A, A1, 128, 128, NULL, 0, 1, 0, A, A, S) == N.NV_ERR_ALIGN


def test_gemm_rows_and_s2f6_epilogue_validation(L):
    f = L.grouped_gemm_nvfp4_fwd_rows
    assert f(A, A, A, A, A, A, NULL, 4, 256, 256, 512, A, N.NV_OUT_BF16, S) == N.NV_ERR_ARG   # no groups
    assert f(A, A, A, A, A, A, A, 4, 256, 200, 512, A, N.NV_OUT_BF16, S) == N.NV_ERR_SHAPE   # N % 128
    assert f(A, A, A, A, A, A, A, 4, 256, 256, 384, A, N.NV_OUT_BF16, S) == N.NV_ERR_SHAPE   # K % 256
    assert f(A, A, A, A, A, A, A, 4, 256, 256, 512, A16, N.NV_OUT_BF16, S) == N.NV_ERR_ALIGN  # y 32-byte
    assert f(A, A, A, A, A, A, A, 4, 256, 256, 512, A, 9, S) == N.NV_ERR_ARG                 # output type
    g = L.grouped_gemm_nvfp4_fwd_swiglu_rows
    assert g(A, A, A, A, A, A, A, 4, 256, 192, 512, A, A, A, S) == N.NV_ERR_SHAPE              # I % 128
    assert g(A, A, A, A, A, A, A, 4, 256, 128, 512, A, A, NULL, S) == N.NV_ERR_ARG             # no h scales
    h = L.grouped_gemm_nvfp4_fwd_rht_s2f6
    assert h(A, A, A, A, A, A, A, 4, 256, 256, 512, 7, NULL, A16, A, S) == N.NV_ERR_ALIGN      # codes 32-byte
    assert h(A, A, A, A, A, A, A, 4, 256, 256, 512, 7, NULL, NULL, A, S) == N.NV_ERR_ARG       # no codes
    assert h(A, A, A, A, A, A, A, 4, 256, 96, 512, 7, NULL, A, A, S) == N.NV_ERR_SHAPE         # N % 128


def test_rht_s2f6_and_four_over_six_validation(L):
    q = L.rht32_s2f6_quantize
    assert q(A, 4, 48, 0, A, A, S) == N.NV_ERR_SHAPE           # cols % 32
    assert q(A16, 4, 64, 0, A, A, S) == N.NV_ERR_ALIGN         # x 32-byte
    assert q(A, 4, 64, 0, A16, A, S) == N.NV_ERR_ALIGN         # codes 32-byte
    assert q(A, 0, 64, 0, A, A, S) == N.NV_OK                  # empty
    d = L.s2f6_dequantize_rht32_inverse
    assert d(A, A, 4, 64, 0, A, 3, S) == N.NV_ERR_ARG          # output type
    assert d(A, A, 4, 64, 0, A16, N.NV_OUT_FP32, S) == N.NV_ERR_ALIGN
    f = L.nvfp4_quantize_four_over_six
    assert f(A, 1, 128, 120, NULL, 0, A, A, A, A, A, 1 << 20, S) == N.NV_ERR_SHAPE   # cols % 16
    assert f(NULL, 1, 128, 128, NULL, 0, A, A, A, A, A, 1 << 20, S) == N.NV_ERR_ARG
    assert f(A, 1, 0, 128, NULL, 0, A, A, A, A, A, 1 << 20, S) == N.NV_OK
    g = L.nvfp4_quantize_requant_four_over_six
    assert g(A, 1, 128, 192, NULL, 0, A, A, A, A, A, 1 << 20, 1, 0, A, A, S) == N.NV_ERR_SHAPE  # cols % 128


def test_fwd_with_bf16_activations_validation(L):
    f = L.grouped_gemm_nvfp4_fwd
    M, N_, K, E = 256, 256, 512, 4
    need = N.nvfp4moe_fwd_workspace_bytes(M, K, E)
    assert need >= M * K // 2 + N.nvfp4moe_scale_bytes(N.nvfp4moe_padded_cap(M, E), K // 16)
    assert N.nvfp4moe_fwd_workspace_bytes(-1, K, E) == 0
    # quantized activations missing without bf16 ones
    assert f(NULL, A, NULL, A, A, A, A, A, E, M, N_, K, A, N.NV_OUT_BF16, NULL, 0, S) == N.NV_ERR_ARG
    # bf16 activations: the workspace must be large enough and aligned
    assert f(A, NULL, NULL, NULL, A, A, A, A, E, M, N_, K, A, N.NV_OUT_BF16, A, need - 1, S) == N.NV_ERR_WORKSPACE
    assert f(A, NULL, NULL, NULL, A, A, A, A, E, M, N_, K, A, N.NV_OUT_BF16, A4, need, S) == N.NV_ERR_WORKSPACE
    assert f(A4, NULL, NULL, NULL, A, A, A, A, E, M, N_, K, A, N.NV_OUT_BF16, A, need, S) == N.NV_ERR_ALIGN


def test_outer_scale_validation(L):
    f = L.nvfp4_outer_scale
    ws = N.nvfp4moe_quantize_workspace_bytes(2, 1, 4096)
    assert f(NULL, 2, 4096, A, A, ws, S) == N.NV_ERR_ARG
    assert f(A, 2, 4100, A, A, ws, S) == N.NV_ERR_SHAPE        # n % 8
    assert f(A4, 2, 4096, A, A, ws, S) == N.NV_ERR_ALIGN
    assert f(A, 2, 4096, A, A, ws - 1, S) == N.NV_ERR_WORKSPACE


def test_selftest_spins_are_bounded(L):
    f = L.nvfp4moe_selftest_wait_timeout
    assert f(0, S) == N.NV_ERR_ARG                  # no iterations
    assert f((1 << 20) + 1, S) == N.NV_ERR_ARG      # above the limit: refused before any launch
    assert f(1 << 40, S) == N.NV_ERR_ARG


def test_noalloc_reports_argument_errors_like_the_workspace_entry_point(L):
    # a shape too large for the fixed scratch AND a bad argument: the argument
    # error wins, exactly as nvfp4_quantize reports it
    big = (1024, 16384, 256)
    assert N.nvfp4moe_quantize_workspace_bytes(*big) > 524288
    q, qn = L.nvfp4_quantize, L.nvfp4_quantize_noalloc
    for args, want in [((NULL,) + big, N.NV_ERR_ARG),                    # no x
                       ((A, 1024, 16384, 248), N.NV_ERR_SHAPE),           # cols % 16
                       ((A4,) + big, N.NV_ERR_ALIGN)]:                    # x not 16-byte aligned
        assert qn(*args, NULL, 0, NULL, A, A, A, S) == want
        assert q(*args, NULL, 0, NULL, A, A, A, A, 1 << 30, S) == want
    assert qn(A, *big, NULL, 0, NULL, A, NULL, A, S) == N.NV_ERR_ARG      # no codes
    assert qn(A, *big, NULL, 0, NULL, A, A, A, S) == N.NV_ERR_WORKSPACE   # valid, too large
    assert qn(A, 1, 0, 256, NULL, 0, NULL, A, A, A, S) == N.NV_OK         # empty: nothing launched


def test_gemm_wait_limit_range(L):
    f = L.nvfp4moe_set_gemm_wait_limit
    assert f(-1) == N.NV_ERR_ARG
    assert f((1 << 26) + 1) == N.NV_ERR_ARG
    assert f(0) == N.NV_OK          # the default


def test_quantize_requant_gather_validation(L):
    f = L.nvfp4_quantize_requant_gather
    ws = 1 << 20
    # x, row_src, src_rows, rows, cols, groups, ngroups, sg_in, sg_out, codes, scales, ws, ws_bytes, seed, off, oc, os
    assert f(A, NULL, 64, 128, 128, A, 2, NULL, A, A, A, A, ws, 1, 0, A, A, S) == N.NV_ERR_ARG      # no row map
    assert f(A, A, 64, 128, 128, NULL, 0, NULL, A, A, A, A, ws, 1, 0, A, A, S) == N.NV_ERR_ARG      # groups required
    assert f(A, A, 64, 128, 192, A, 2, NULL, A, A, A, A, ws, 1, 0, A, A, S) == N.NV_ERR_SHAPE       # cols % 128
    assert f(A, A1, 64, 128, 128, A, 2, NULL, A, A, A, A, ws, 1, 0, A, A, S) == N.NV_ERR_ALIGN      # row map 4-byte
    assert f(A, A, 64, 128, 128, A, 2, NULL, A, A, A, A, 16, 1, 0, A, A, S) == N.NV_ERR_WORKSPACE   # no room
    # a given outer scale still needs room for the tokens' codes (src_rows <= rows)
    assert f(A, A, 64, 128, 128, A, 2, A, A, A, A, NULL, 0, 1, 0, A, A, S) == N.NV_ERR_WORKSPACE
    assert f(A, A, 64, 0, 128, A, 2, NULL, A, A, A, A, ws, 1, 0, A, A, S) == N.NV_OK                # empty


def test_quantize_gather_workspace_bytes():
    def r256(n):
        return (max(n, 1) + 255) // 256 * 256
    for src, rows, cols in ((16384, 131072, 4096), (1000, 64, 256), (0, 128, 128), (300, 300, 128)):
        want = N.nvfp4moe_quantize_workspace_bytes(1, rows, cols) + (src * 4 + 255) // 256 * 256
        if src <= rows:  # the tokens' NVFP4 codes and batched scales
            want += r256(src * cols // 2) + r256(N.nvfp4moe_scale_bytes((src + 127) // 128 * 128, cols // 16))
        assert N.nvfp4moe_quantize_gather_workspace_bytes(src, rows, cols) == want
    assert N.nvfp4moe_quantize_gather_workspace_bytes(-1, 128, 128) == 0
