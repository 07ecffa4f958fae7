"""Causal grouped-query FlashAttention, forward and backward, for GB300 (sm_103a).

The compute path is the CUDA library ``libnea_attn.so`` built from ``csrc/``;
``nea`` is its thin ctypes binding (argument marshalling only).
"""
