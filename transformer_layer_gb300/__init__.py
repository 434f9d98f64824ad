"""GB300-native fused transformer-layer decode (C-ABI library + thin binding).

The compute path lives in ``libdslayer.so`` (CUDA for sm_103a, built by
``transformer_layer_gb300.build``).  ``transformer_layer_gb300.ds`` holds the
ctypes binding with the same names as the C entry points.  The library is
loaded on first use of the binding; if it is missing the binding raises, and
there is no CPU fallback.
"""
__all__ = ["ds", "inputs", "workloads"]
