"""GB300-native fused FP8 attention forward (E4M3 Q/K/V, bf16/fp16 O, fp32 LSE).

The compute path is the C-ABI library ``libfa8.so`` (hand-written CUDA for sm_103a);
``fp8_attention_forward_gb300.fa8`` is its thin ctypes binding.
"""
__all__ = ["fa8", "inputs"]
