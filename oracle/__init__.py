"""CPU oracle for the NVFP4-forward / MXFP8-backward expert numerics.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the pages of "End-to-End 4-Bit Training" (Thinking
Machines Lab) compute on the expert hot path.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The CUDA library never calls it and
shares no code with it; the only module both sides use is the seeded input
generator ``precision_moe_numerics_nvfp4_gb300.workloads``, which holds none of
the method's arithmetic.

Floating point follows the pages' precision where they fix it (the E2M1,
E4M3 and E8M0 grids, the FP32 outer scale) and the conventions stated in each
function's docstring where they do not; everything else is float64.  Rounding
to a grid is done by brute-force nearest search over the enumerated grid, not
by bit tricks.

Modules
-------
formats   E2M1 / E4M3 / E8M0 decoding from their bit fields; RN and SR to a grid
philox    Philox4x32-10 counter-based generator and the per-element bit draw
nvfp4     NVFP4 1x16 quantize / dequantize, 16x16 tile and 16x1 column variants
mxfp8     MXFP8 1x32 quantize (RN or SR) with E8M0 scales
requant   dequantize -> transpose -> SR re-quantize NVFP4 -> MXFP8
layout    the block-scaled MMA scale-factor layout (128x4 atoms) as an index map
gemm      FP64 grouped GEMM references over dequantized operands and the bound
swiglu    SwiGLU forward / backward between the two expert GEMMs

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
except where its docstring says "parity unpinned".
"""
