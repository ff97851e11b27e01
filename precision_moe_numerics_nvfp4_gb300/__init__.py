"""GB300 (sm_103a) NVFP4-forward / MXFP8-backward expert numerics.

The compute lives in the C-ABI library ``libnvfp4moe.so`` built from
``csrc/``; ``precision_moe_numerics_nvfp4_gb300.nvfp4moe`` is its thin ctypes
binding.  ``workloads`` draws the seeded synthetic inputs.
"""
