"""Block-scaled FP8 linear projection for NVIDIA GB300 (sm_103a).

Modules:
  bfp8   ctypes binding of libbfp8.so (include/bfp8.h), same names as the C ABI.
  build  compiles libbfp8.so in-tree with nvcc for sm_103a.
  synth  seeded synthetic inputs (random draws only).

Importing the package itself loads nothing. ``from block_scaled_fp8_token_gb300
import bfp8`` loads the CUDA library and fails loudly if it is missing.
"""
