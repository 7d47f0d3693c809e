"""GB300-native exact fused attention, forward and backward (sm_103a).

The compute path is the C-ABI library ``libattn.so`` built from ``csrc/``;
``exact_attention_86_gb300.attn`` is its thin Python binding.  Importing the
package does not load the library; the first call into ``attn`` does, and
raises if the library is missing (there is no CPU fallback).
"""
