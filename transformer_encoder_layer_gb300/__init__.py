"""GB300 (sm_103a) forward pass of a masked post-LN transformer encoder stack.

The compute runs in hand-written CUDA kernels behind the C ABI declared in
``include/tl_encoder.h``; :mod:`.binding` marshals torch tensors to it.
Importing the package does not load the library; ``binding.load()`` does, and
raises if it has not been built.
"""
__all__ = ["inputs", "gate"]
