"""GB300-native single-query decode attention (split-KV, LSE merge, GQA packing, paged
KV cache, unified-max softmax with synchronised recompute) behind a small C ABI.

The CUDA library is loaded on first use by `decode_attention_attn_gb300.binding`; a
missing or unbuilt library raises there, loudly. There is no CPU fallback.
"""
__all__ = ["binding", "workloads"]
