"""nvfp4kv: NVFP4 paged KV cache for one GB300 (sm_103a).

The compute lives in the CUDA library ``libnvfp4kv.so`` (see
``include/nvfp4kv.h``); this package is a thin ctypes binding over it plus
seeded workload generators (``inputs``).
"""
