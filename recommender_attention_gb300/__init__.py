"""GB300-native HSTU attention forward.

The compute path is the C-ABI library ``libhstu_attn.so`` (hand-written
sm_103a CUDA) built in-tree; :mod:`recommender_attention_gb300.hstu` is a thin
ctypes binding over it.  Importing the package does not load the library; the
first call does, and fails loudly when it is missing.
"""
__all__ = ["hstu", "workloads"]
