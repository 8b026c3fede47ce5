"""GB300-native (sm_103a) chunked forward pass of Kimi Delta Attention (KDA).

The compute lives in libkda.so (hand-written CUDA behind the C ABI of
include/kda.h); this package is its thin Python binding plus the seeded
synthetic workloads. Importing the package does not load the library: the
first call does, and fails loudly if libkda.so has not been built.
"""
from .kda import (fwd, fwd_noalloc, NOALLOC_MAX_SCRATCH, workspace_size, debug_chunk_matrices, device_status,  # noqa: F401
                  max_chunks, plan, CP_OFF, CP_SEGMENTS)

__version__ = "0.1.0"
