"""GB300-native Mamba-2 SSD layer (chunked selective scan, forward and
backward) behind a C ABI (include/ssd.h, libssd.so).

Submodules:
  inputs     seeded synthetic inputs of the layer workloads (no arithmetic)
  build_ext  builds libssd.so in-tree with nvcc for sm_103a
  _lib       ctypes binding of the C ABI (raises if libssd.so is missing)
  runner     device buffers of one problem and the calls through the C ABI
"""
__all__ = ["inputs", "build_ext"]
