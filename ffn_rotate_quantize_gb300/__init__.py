"""Rotated-INT8 linear layers, SwiGLU FFN and dx backward for GB300 (sm_103a).

The compute path is the C-ABI library ``libgbq.so`` (hand-written CUDA).
``ffn_rotate_quantize_gb300.ops`` is the thin Python binding over it.
"""
