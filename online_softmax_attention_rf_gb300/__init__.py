"""Fused online-softmax attention for one GB300 (sm_103a).

The compute path lives in ``librf.so`` (CUDA kernels behind a C ABI declared
in ``include/rf.h``); ``api`` is a thin ctypes binding that only marshals
torch tensors into pointers and sizes. There is no CPU fallback: every call
fails loudly if the library is missing.
"""
