"""QLoRA NF4 linear-layer hot path for the B300 (sm_103a).

The compute lives in ``libqlora_b300.so`` (CUDA kernels behind the C ABI of
``include/qlora.h``); this package is its thin Python binding plus the
seeded synthetic input generators.  Build with
``python -m bit_nf4_quantized_35_b300.build``.
"""
from .capi import (NF4Weight, QloraError, Workspace, dequant, linear_bwd, linear_fwd,  # noqa: F401
                   load, nf4_codebook, nf4_sizes, nf4_thresholds, quantize_nf4, workspace_size)
