"""GB300-native hybrid Gated-DeltaNet + sink/sliding-window softmax layer.

The compute path is the C-ABI library ``libhla.so`` (hand-written sm_103a CUDA
kernels); ``linearized_attention_rope_gb300.hla`` is its thin ctypes binding.
"""
