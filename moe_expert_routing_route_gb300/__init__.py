"""GB300-native (sm_103a) single-GPU MoE layer hot path.

top-k routing -> init-routing permutation -> grouped SwiGLU expert GEMM on
tcgen05 tensor cores -> finalize-routing with the shared expert added.

The compute lives in ``libmoe.so`` (CUDA, C ABI declared in ``include/moe.h``).
``moe_expert_routing_route_gb300.binding`` is a thin ctypes layer over it; it
raises if the library is missing -- there is no CPU fallback.
"""
