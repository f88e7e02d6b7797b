"""GB300-native causal streaming-softmax attention (forward and split backward).

The compute path is a C-ABI CUDA library (``libattn.so``, sm_103a) whose
entry points ``attn_fwd``, ``attn_row_terms``, ``attn_bwd_keys`` and
``attn_bwd_queries`` are bound in :mod:`causal_streaming_softmax_gb300.api`.
Importing this package does not load the library; the first call does, and
fails loudly if it is missing.
"""
__version__ = "0.1.0"
