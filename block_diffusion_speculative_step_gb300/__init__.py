"""GB300-native DFlash block-diffusion speculative decoding: one
draft-and-verify cycle on hand-written sm_103a CUDA kernels behind a C ABI.

Submodules:
  dflash  -- thin ctypes binding of the C ABI (same names as include/dflash.h)
  engine  -- device buffers and the per-cycle call sequence
  synth   -- seeded synthetic inputs (no arithmetic of the method)
  build   -- compiles the CUDA library in-tree
"""
__all__ = ["dflash", "engine", "synth", "build"]
