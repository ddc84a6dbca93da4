"""Vocab-parallel cross-entropy for GB300 (sm_103a).

The compute path is the C-ABI library ``libvpce.so`` (hand-written CUDA
kernels, see ``csrc/``); :mod:`vocab_sharded_lm_gb300.vpce` is its thin ctypes
binding.  Importing this package loads nothing; the binding loads the library
on first use and raises if it is missing.
"""
__all__ = ["vpce", "synth"]
