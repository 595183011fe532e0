"""GB300-native routed-expert MoE forward.

The compute path is the C-ABI library ``libmoe_routed_gb300.so`` (hand-written
sm_103a CUDA kernels).  :mod:`.binding` is its thin Python binding; importing
it loads the library and fails loudly when it has not been built.
"""

__all__ = ["binding", "workloads", "roofline"]
