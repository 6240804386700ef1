"""GB300-native 2-bit sign-symmetric MoE experts (vLLM-Moet's moe_w2 layer).

Modules:
  moe_w2  ctypes binding of libmoe_w2.so (the CUDA library; C ABI in include/moe_w2.h)
  build   nvcc build of the library for sm_103a
  inputs  seeded synthetic inputs (no layer arithmetic)

Importing the package loads nothing; ``moe_w2.load()`` opens the library.
"""
