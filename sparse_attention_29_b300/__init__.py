"""libdsa: the DeepSeek Sparse Attention hot path for one B300 (sm_103a).

lightning indexer -> causal top-k -> sparse MLA (MQA / absorbed mode), with IndexShare
reuse of one index set across a group of layers and an optional paged cache.

The compute lives in the C-ABI library libdsa.so (CUDA kernels, see csrc/); the Python
module `capi` is a thin ctypes binding over it.  Importing this package loads nothing:
`inputs` (seeded synthetic workloads) works without a GPU.
"""
__all__ = ["inputs", "capi", "pipeline"]
