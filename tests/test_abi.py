"""The C-ABI library builds, loads and exports every function the header
declares; its host-only helpers agree with the oracle's layout restatement.
No GPU work is done here."""
import numpy as np
import pytest

from oracle import layout as L
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N


@pytest.fixture(scope="module")
def lib():
    from precision_moe_numerics_nvfp4_gb300 import build
    build.build()
    return N.lib()


def test_exports_every_declared_function(lib):
    names = N.declared_functions()
    assert len(names) >= 16
    for n in ["nvfp4_quantize", "dequant_transpose_requant_sr", "grouped_gemm_nvfp4_fwd",
              "grouped_gemm_mxfp8_dx", "grouped_gemm_mxfp8_dw", "mxfp8_quantize"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in N._SIGS, f"binding lacks {n}"


def test_scale_offset_matches_oracle_layout(lib):
    for kblocks in (1, 4, 7, 16, 33):
        for rp in (0, 1, 31, 32, 63, 64, 127, 128, 300, 1025):
            for c in range(kblocks):
                assert N.nvfp4moe_scale_offset(rp, c, kblocks) == int(L.atom_offset(rp, c, kblocks))


def test_padded_cap_and_sizes(lib):
    for M, E in ((0, 1), (428, 4), (131072, 64), (2048, 128), (1, 1)):
        assert N.nvfp4moe_padded_cap(M, E) == L.padded_cap(M, E)
    assert N.nvfp4moe_scale_bytes(300, 7) == L.scale_buffer_bytes(300, 7)
    o = np.array([0, 5, 5, 300, 428])
    assert L.group_padded_starts(o)[-1] <= N.nvfp4moe_padded_cap(428, 4)


def test_status_strings(lib):
    assert N.status_string(0) == "ok"
    assert N.status_string(N.NV_ERR_TIMEOUT) == "bounded wait ran out"
    assert "sm_103a" in N.nvfp4moe_version()


def test_gemm_kernel_choice_is_validated(lib):
    for v in (N.GEMM_ONE_PER_SM, N.GEMM_TWO_PER_SM, N.GEMM_CTA_PAIR, N.GEMM_CTA_PAIR_N128, N.GEMM_AUTO):
        N.nvfp4moe_set_gemm_kernel(v)
    for bad in (-1, 5, 99):
        with pytest.raises(N.NvError):
            N.nvfp4moe_set_gemm_kernel(bad)
