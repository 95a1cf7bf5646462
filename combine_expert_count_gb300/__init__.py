"""libmoeroute: MoE expert-parallel dispatch and combine on one GB300.

The compute path is the CUDA library ``libmoeroute.so`` (C ABI in
``include/moeroute.h``); ``moeroute`` is its Python binding and
``workloads`` synthesises seeded inputs.  Importing this package does not
load the library; the first call into ``moeroute`` does, and raises if it has
not been built.
"""
__all__ = ["moeroute", "workloads", "build"]
