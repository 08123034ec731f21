"""Emulated-rank gradient collectives for one GB300 GPU.

The compute path lives in ``libcr.so`` (CUDA kernels for sm_103a behind the C
ABI declared in ``include/cr.h``); ``fsdp_emulated_ranks_gb300.cr`` is a thin
ctypes binding with the same entry-point names.  Importing this package loads
nothing: the library is opened on first use and a missing library raises.
"""

__all__ = ["cr", "inputs"]
