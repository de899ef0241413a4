"""B300-native KV-cache compression hot path: score -> select -> compact -> decode.

The compute runs in hand-written CUDA kernels for sm_103a behind a C ABI
(``include/kvc.h``, ``libkvc.so``).  ``binding`` is the thin ctypes layer that
marshals torch tensors into that ABI; it is imported on demand so that the
input generators can be used without a GPU.
"""
__all__ = ["binding", "inputs"]
