"""Block-wise masked-diffusion decoding on B300 (sm_103a).

The compute path is libdd.so (C-ABI in include/dd.h, CUDA sources in csrc/).
`binding` is the ctypes layer with the C names; `decoder` wraps it for torch
tensors.  Importing this package does not load the library; the first call
does, and fails loudly if it has not been built.
"""

__all__ = ["binding", "decoder", "build"]
