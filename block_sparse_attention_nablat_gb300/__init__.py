"""NABLA (Neighborhood-Adaptive Block-Level Attention) for GB300 (sm_103a).

The compute lives in hand-written CUDA kernels behind the C ABI declared in
include/nabla.h (library libnabla.so, built in-tree by __graft_entry__.build()).
`nabla` is the thin ctypes binding; `workloads` holds the seeded synthetic inputs.
"""
