"""GB300-native GQA decode attention over a paged KV cache.

``gqa_paged_kv_gb300.qdec`` is the Python binding of libqdec (the C ABI in
include/qdec.h, CUDA kernels for sm_103a in csrc/); ``build`` compiles it;
``workloads`` generates seeded synthetic decode inputs.  The binding is not
imported here so that input generation works on machines without the
compiled library.
"""
__all__ = ["build", "qdec", "workloads"]
