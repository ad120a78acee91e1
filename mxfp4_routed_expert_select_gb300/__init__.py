"""GB300 (sm_103a) MXFP4 routed-expert MoE layer.

The compute lives in ``libk3moe.so`` (hand-written CUDA behind the C ABI of
``include/k3moe.h``); ``k3moe`` is its ctypes binding.  Build with
``__graft_entry__.build()`` (or ``python -m mxfp4_routed_expert_select_gb300._build``).
"""
from . import k3moe  # noqa: F401
