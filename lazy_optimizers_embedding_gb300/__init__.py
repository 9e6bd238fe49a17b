"""lazy_optimizers_embedding_gb300 -- the sparse / lazy optimizer step for large
fp32 embedding tables on one GB300 (sm_103a).

The compute path is the C-ABI library ``libsparseopt.so`` (hand-written CUDA
kernels; header ``include/sparseopt.h``).  ``binding`` is its thin ctypes
binding (same entry-point names); ``workloads`` draws seeded synthetic inputs.
Importing the package does not load the library; ``from
lazy_optimizers_embedding_gb300 import binding`` does, and raises if the library
has not been built (``__graft_entry__.build()``).
"""
