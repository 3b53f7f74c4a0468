"""GB300-native Qwen3-0.6B-shaped decoder forward pass (prefill + KV-cached decode).

The CUDA library and its ctypes binding live in :mod:`transformer_decode_qwen3_gb300.binding`;
importing this package loads nothing native.
"""
