"""Single-GPU MoE token dispatch, grouped int8 expert FFN and weighted combine
for GB300 (sm_103a).

The compute runs in hand-written CUDA kernels behind a C ABI
(``libmoe_gb300.so``, declared in ``include/moe_gb300.h``).  The Python layer
only marshals pointers, sizes and streams; PyTorch provides device memory and
streams.  Importing this package does not load the library; the first call
through :mod:`combine_route_count_prefix_gb300.binding` does, and it raises if
the library was not built.
"""

__all__ = ["binding", "workloads"]
