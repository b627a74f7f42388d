"""fp4idx for GB300: the fused FP4 indexer pre-pass of a DeepSeek-style
sparse-attention indexer, as hand-written CUDA for sm_103a behind a C ABI.

Submodules:
  fp4idx     -- ctypes binding of libfp4idx.so (loads the CUDA library on
                import and raises if it is missing: there is no CPU path).
  build      -- compiles libfp4idx.so with nvcc for sm_103a.
  workloads  -- seeded synthetic inputs (no arithmetic of the method).
"""
__all__ = ["fp4idx", "build", "workloads"]
