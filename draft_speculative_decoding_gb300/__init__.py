"""GB300-native draft-block select-and-verify for DFlash 2 block drafting.

Submodules:
  binding    -- ctypes binding to the C-ABI CUDA library (libdfs.so); loads lazily
  workloads  -- seeded synthetic inputs shaped like the pages' workloads
  build      -- compiles the CUDA library for sm_103a
"""
