"""CSA2 (Compressed Sparse Attention 2) attention step for one GB300 GPU.

The computation runs in ``libcsa2.so`` (hand-written CUDA for sm_103a, C ABI
in ``include/csa2.h``); :mod:`.csa2` is its Python binding, :mod:`.device`
sets up synthetic workloads on the device and drives the layer pattern.
"""
__all__ = ["csa2", "synth", "workloads", "build"]
