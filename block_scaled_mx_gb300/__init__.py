"""GB300-native MX block-scaled sparse-MoE expert layer.

The compute path is the C-ABI library ``libmxmoe.so`` (hand-written CUDA for
sm_103a); ``block_scaled_mx_gb300.mxmoe`` is its thin ctypes binding and
``block_scaled_mx_gb300.workload`` draws the seeded synthetic inputs.  Importing
the package does not load the library; the first call through the binding does,
and raises if the library is missing.
"""
__all__ = ["mxmoe", "workload"]
