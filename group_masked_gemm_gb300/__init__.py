"""GB300-native (sm_103a) group-masked GEMMs for WIDE token-level dynamic
width pruning: mask reordering, GEMM-MN (gate/up with fused SiLU, q_proj)
and GEMM-K (down_proj, o_proj), prefill and decode.

The compute runs in ``libwide.so`` (hand-written CUDA, C ABI declared in
``include/wide.h``); ``ops`` is a thin ctypes binding over it.  Importing
the package does not load the library; the first op call does, and fails
loudly if the library is missing.
"""

__all__ = ["ops", "synthetic"]
