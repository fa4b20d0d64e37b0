"""GB300 (sm_103a) Megatron-style transformer layer: forward, backward and the
vocab-chunked tied-embedding cross-entropy, as a C-ABI CUDA library
(libmgb.so, include/mgb.h) with a thin ctypes binding (`mgb`).

`inputs` holds the seeded synthetic workloads; `runner` allocates device
buffers with PyTorch and calls the library.
"""
__version__ = "0.1.0"
