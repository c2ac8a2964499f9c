"""GQA fused attention for one GB300 (sm_103a): split-KV decode and causal prefill.

The compute lives in ``libgqa_attn.so`` (hand-written CUDA, C ABI declared in
``include/gqa_attn.h``). ``gqa_attention_split_gb300.api`` is a ctypes
binding with the same entry-point names; it only marshals arguments. Importing
this package does not load the library; the first call does, and raises if
the library has not been built.
"""
