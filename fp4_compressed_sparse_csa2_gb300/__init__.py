"""GB300-native CSA2 attention layer (DeepSeek-V4.1-Flash) over an FP4 KV cache.

The compute path is libcsa2.so (hand-written sm_103a CUDA behind the C ABI in
include/csa2.h); ``fp4_compressed_sparse_csa2_gb300.csa2`` is its thin ctypes binding.
``fp4_compressed_sparse_csa2_gb300.build`` compiles the library in-tree with nvcc.
"""
