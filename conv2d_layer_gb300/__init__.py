"""GB300-native (sm_103a) conv2d training step: C-ABI CUDA library + thin binding.

Submodules:
  abi        ctypes binding of include/conv2d.h (same names as the C entry points)
  layer      Conv2dLayer: torch-owned buffers around the ABI calls
  workloads  seeded synthetic inputs (shared with the test oracle)
  build      in-tree nvcc build of libconv2d.so for sm_103a

Importing the package does not load the CUDA library; the first ABI call does,
and fails loudly if it cannot be loaded or built.
"""
