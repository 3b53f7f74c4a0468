"""CPU oracles for the Qwen3-0.6B decoder forward pass and sampler.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import this package; the product path never does.
It shares no code with the CUDA library: its only input dependency is the
seeded generator module (transformer_decode_qwen3_gb300.synth).

  qwen3_ref.c / qwen3_c.py  plain single-precision C (float storage, double
                            accumulators, OpenMP), through ctypes
  qwen3_ref.py              the same definition in numpy float64, the cross-check
"""
