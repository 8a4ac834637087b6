"""Gated DeltaNet linear-attention layer for one NVIDIA GB300 (sm_103a).

Modules:
  build    -- nvcc build of the in-tree CUDA library libgdn.so
  binding  -- ctypes binding of the C ABI (include/gdn.h), same entry-point names
  synth    -- seeded synthetic inputs (random draws only; no layer arithmetic)
"""
