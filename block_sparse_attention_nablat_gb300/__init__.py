"""NABLA (Neighborhood-Adaptive Block-Level Attention) for GB300 (sm_103a).

The compute lives in hand-written CUDA kernels behind the C ABI declared in
include/nabla.h (library libnabla.so, built in-tree by __graft_entry__.build()):
the nablaT_v2 mask builder and the block-sparse attention forward (with an
optional log-sum-exp output), the attention backward, the top-k block selector,
the fractal token order and the STA window.  `nabla` is the thin ctypes binding;
`workloads` holds the seeded synthetic inputs.
"""
