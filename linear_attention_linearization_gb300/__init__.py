"""GB300-native STILL intra-layer hybrid attention (sm_103a).

``still``   -- Python binding of the C-ABI library ``libstill.so`` (argument
               marshalling only; every step of the layer runs in its kernels).
``inputs``  -- seeded synthetic inputs shaped like the pages' workloads.
``build``   -- compiles the CUDA library in-tree with nvcc for sm_103a.

Submodules are imported on demand so that ``inputs`` stays usable on hosts
without a GPU.
"""
__all__ = ["still", "inputs", "build"]
