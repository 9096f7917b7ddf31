"""GB300 (sm_103a) FlashAttention-2 forward: C-ABI CUDA library + Python binding.

The compute path is the CUDA library ``libfa2.so`` built from ``csrc/``; the
Python module :mod:`attention_fa2_forward_03_gb300.fa2` only marshals
arguments to its C entry points. There is no Python or CPU fallback.
"""
__version__ = "0.3.0"
