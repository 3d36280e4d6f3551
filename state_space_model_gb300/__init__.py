"""Mamba-2 SSD chunked forward for GB300 (sm_103a).

The compute runs in the C-ABI library ``libssd_gb300.so`` (hand-written CUDA
kernels); :mod:`state_space_model_gb300.ssd` is its thin Python binding.
Importing this package does not load the library; the first call does, and
fails loudly if it has not been built.
"""

__all__ = ["ssd", "inputs"]
