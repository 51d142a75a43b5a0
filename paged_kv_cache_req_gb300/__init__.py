"""Attention over a paged KV cache on one GB300 GPU (sm_103a).

The compute lives in ``libpkv.so`` (hand-written CUDA behind the C ABI of
``include/pkv.h``); ``_binding`` is its ctypes binding, ``engine.DecodeStep``
the per-step API, ``workloads`` the seeded synthetic inputs, and ``build`` the
nvcc build of the library.  Importing the package does not load the library;
importing ``_binding`` or ``engine`` does, and fails loudly if it is missing.
"""
__all__ = ["build", "workloads"]
