"""GB300-native SiTU routed-MoE expert layer on block-scaled FP4 weights.

The compute path lives in the CUDA library built from ``csrc/``
(``libsitu_moe.so``, C ABI declared in ``include/situ_moe.h``); ``binding``
marshals arguments to it through ctypes.  ``workloads`` draws the seeded
synthetic inputs.  Importing this package loads nothing: the library is
loaded on first use by ``binding``.
"""
__all__ = ["binding", "workloads", "build"]
