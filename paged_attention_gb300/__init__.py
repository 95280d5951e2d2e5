"""GB300-native paged-KV-cache attention forward (sm_103a).

The compute path lives in the C-ABI shared library built from ``csrc/``
(declared in ``include/pa.h``); :mod:`paged_attention_gb300.binding` is a
thin ctypes binding with the same names.  PyTorch is used for device memory
and streams only.  Importing this package does not load the CUDA library;
the first call into the binding does, and fails loudly if it is missing.
"""
__all__ = ["binding", "workloads"]
