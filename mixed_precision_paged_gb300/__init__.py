"""GB300-native mixed-fidelity paged KV attention (FP16 keys, FP16/E4M3 values).

The compute path is the ``ekv`` CUDA library (hand-written sm_103a kernels behind a
C ABI, declared in ``include/ekv.h``); ``mixed_precision_paged_gb300.ekv`` is its thin
ctypes binding. Importing the binding fails loudly when the library is not built.
"""

__all__ = ["ekv", "workloads", "roofline", "build"]
