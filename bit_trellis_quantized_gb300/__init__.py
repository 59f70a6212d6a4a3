"""GB300 (sm_103a) library for the Escha-W2 trellis MoE expert path.

The compute lives in ``libescha.so`` (CUDA kernels behind the C ABI of
``include/escha.h``); ``native`` is its Python binding.
"""
__all__ = ["native"]
