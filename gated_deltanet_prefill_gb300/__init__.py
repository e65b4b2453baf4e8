"""GB300-native (sm_103a) Gated DeltaNet-2 chunked prefill forward.

The compute path is the CUDA library ``libgdn2.so`` built from ``csrc/``;
``gdn2`` is its thin ctypes binding.  Importing this package loads nothing:
the library is opened on first use and a missing library is an error.
"""
__all__ = ["gdn2", "inputs"]
