"""The algorithmic bytes behind bench.py's roofline figures, recounted from the tensors.

The bench states the bytes a decode step must move in closed form (layer parameter counts,
norm widths, cache bytes per position).  These tests count the same bytes a second way, from
the checkpoint's own tensor list (names and shapes as the article's Step 5-8 code names them),
so that a dropped term or a wrong width in the closed form fails here on the CPU.
"""
import math

import bench
from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth

S = synth.QWEN3_0_6B


def _shapes():
    return synth.weight_shapes(S)


def test_bf16_weight_bytes_equal_the_checkpoint():
    # every tensor once in bf16; the LM head is the embedding (tied), so it is not counted twice
    total = sum(2 * math.prod(shp) for shp in _shapes().values())
    assert bench.WEIGHT_BYTES == total
    assert abs(total - 1.19e9) < 0.01e9          # the 1.19 GB the documentation quotes
    assert 2 * S.vocab * S.hidden == 311_164_928  # the LM head's share (311.2 MB)


def test_int8_weight_bytes_equal_codes_scales_and_norms():
    # quantised matrices (and the tied embedding): one byte per weight and one fp32 scale per
    # output channel (row); norm weights stay bf16
    total = 0
    for name, shp in _shapes().items():
        if name == "model.embed_tokens.weight" or name.endswith(R.QUANTISED_SUFFIXES):
            rows, cols = shp
            total += rows * cols + 4 * rows
        else:
            total += 2 * math.prod(shp)
    assert bench.WEIGHT_BYTES_INT8 == total


def test_cache_bytes_per_position():
    # K and V of every layer and KV head, head_dim bf16 values each
    per_layer = 2 * S.n_kv_heads * S.head_dim * 2
    assert bench.KV_LAYER_BYTES_PER_POS == per_layer == 4096
    assert bench.KV_BYTES_PER_POS == S.n_layers * per_layer == 114_688


def test_step_bytes_average_the_cache_over_the_timed_positions():
    # step i (0-based) attends over PROMPT + i + 1 positions (the prompt, the earlier steps and
    # itself); the bench's per-step figure is the mean over the K timed steps
    K = 4
    want = bench.WEIGHT_BYTES + sum((bench.PROMPT + i + 1) for i in range(K)) / K * bench.KV_BYTES_PER_POS
    got = bench.DecodeBs1.bytes_per_step(None, K)
    assert abs(got - want) < 1e-6 * want


def test_prefill_flops():
    # projections: 2 FLOP per weight per token, every layer matrix (q, k, v, o, gate, up, down)
    T, B = bench.PREFILL_T, bench.PREFILL_B
    per_token = 2 * sum(math.prod(shp) for name, shp in _shapes().items() if name.endswith(R.QUANTISED_SUFFIXES))
    linear, attn, head = bench.Prefill.flops(None)
    assert linear == per_token * T * B
    assert abs(linear - 14.43e12) < 0.01e12        # the 14.43 TFLOP per prefill the profiles quote
    # attention: q.k and p.v, 2 * head_dim FLOP each per head and visible (query, key) pair; a
    # causal prompt of T tokens has T (T + 1) / 2 pairs.  The bench counts T^2 / 2 (0.05% fewer).
    pairs = sum(p + 1 for p in range(T))
    exact = 4 * S.head_dim * S.n_heads * pairs * S.n_layers * B
    assert abs(attn - exact) <= exact / T
    # the LM head runs on the last token of each sequence only
    assert head == 2 * S.hidden * S.vocab * B
