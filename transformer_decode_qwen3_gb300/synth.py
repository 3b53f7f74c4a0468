"""Seeded synthetic inputs for the Qwen3-0.6B-shaped decoder.

This module is the only code shared by the CPU oracle and the CUDA path, and it
holds none of the model's arithmetic: it turns (seed, stream, index) into bf16
bit patterns, token ids and cache lengths with a counter-based integer hash.

Every value is produced by exact integer arithmetic plus one IEEE fp32 multiply,
so the same call gives bit-identical results on any torch device (CPU or CUDA)
and on any host architecture.

Recipe (one value per counter):
  h      = mix32(mix32(index XOR k0) XOR k1)     k0, k1 derived from (seed, stream)
  s      = sum of the four bytes of h            Irwin-Hall(4), integer in [0, 1020]
  z      = s - 510                               mean 0, std sqrt(4*(2^16-1)/12)
  value  = bf16_rne(fp32(z) * fp32(std / 147.8...))
so "N(0, std)" draws are approximated by a scaled sum of four uniform bytes.
Norm weights are exactly 1.0.  Token ids are floor(h * V / 2^32).
"""
from __future__ import annotations

import dataclasses
import math

import torch

M32 = 0xFFFFFFFF
_IH4_STD = math.sqrt(4.0 * (256.0 * 256.0 - 1.0) / 12.0)  # std of a sum of 4 uniform bytes

# stream ids: one per generated tensor family
STREAM_EMBED = 0
STREAM_LAYER_BASE = 1          # + 16 * layer + slot
STREAM_TOKENS = 1 << 20        # + call index
STREAM_KV = 2 << 20            # + 2 * layer + (0 for K, 1 for V)
STREAM_LENGTHS = 3 << 20
LAYER_SLOTS = {"q_proj": 1, "k_proj": 2, "v_proj": 3, "o_proj": 4,
               "gate_proj": 5, "up_proj": 6, "down_proj": 7}


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Sizes of a Qwen3 dense decoder (defaults: Qwen3-0.6B)."""
    n_layers: int = 28
    hidden: int = 1024
    n_heads: int = 16
    n_kv_heads: int = 8
    head_dim: int = 128
    intermediate: int = 3072
    vocab: int = 151936
    weight_std: float = 0.02


QWEN3_0_6B = ModelShape()


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """32-bit avalanche mix on int64 tensors holding values in [0, 2^32).

    Both multipliers are below 2^31, so every product stays below 2^63 and no
    signed overflow happens on any device.
    """
    x = x ^ (x >> 16)
    x = (x * 0x7FEB352D) & M32
    x = x ^ (x >> 15)
    x = (x * 0x5BD1E995) & M32
    x = x ^ (x >> 16)
    return x


def _keys(seed: int, stream: int) -> tuple[int, int]:
    t = torch.tensor([(seed * 0x9E3779B1 + stream) & M32, (stream * 0x85EBCA77 + seed + 0x27D4EB2F) & M32],
                     dtype=torch.int64)
    k = _mix32(_mix32(t) ^ 0x165667B1)
    return int(k[0]), int(k[1])


def hash_u32(seed: int, stream: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """n hashed 32-bit values (int64 tensor) for counters start .. start+n-1."""
    if start < 0 or start + n > (1 << 32):
        raise ValueError("counter range must lie in [0, 2^32)")
    k0, k1 = _keys(seed, stream)
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    return _mix32(_mix32(idx ^ k0) ^ k1)


def _fp32_to_bf16_bits(f: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even fp32 -> bf16, returned as int16 bit patterns (finite inputs)."""
    b = f.view(torch.int32).to(torch.int64) & M32
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    b = b & 0xFFFF
    b = torch.where(b >= 0x8000, b - 0x10000, b)
    return b.to(torch.int16)


def normal_bf16(seed: int, stream: int, n: int, std: float, device="cpu",
                start: int = 0, chunk: int | None = None) -> torch.Tensor:
    """n approximately N(0, std) values as a torch.bfloat16 tensor (see module doc)."""
    out = torch.empty(n, dtype=torch.int16, device=device)
    if chunk is None:
        chunk = (1 << 20) if out.device.type == "cpu" else (1 << 24)
    scale = torch.tensor(std / _IH4_STD, dtype=torch.float32).item()
    scale_t = torch.tensor(scale, dtype=torch.float32, device=device)
    for c0 in range(0, n, chunk):
        m = min(chunk, n - c0)
        h = hash_u32(seed, stream, start + c0, m, device)
        pair = (h & 0x00FF00FF) + ((h >> 8) & 0x00FF00FF)   # two 16-bit lanes of byte sums
        s = (pair & 0xFFFF) + (pair >> 16)
        z = (s - 510).to(torch.float32)
        out[c0:c0 + m] = _fp32_to_bf16_bits(z * scale_t)
    return out.view(torch.bfloat16)


def ones_bf16(n: int, device="cpu") -> torch.Tensor:
    return torch.full((n,), 0x3F80, dtype=torch.int16, device=device).view(torch.bfloat16)


def token_ids(seed: int, call: int, n: int, vocab: int, device="cpu") -> torch.Tensor:
    """n token ids uniform in [0, vocab) as int32."""
    h = hash_u32(seed, STREAM_TOKENS + call, 0, n, device)
    return ((h * vocab) >> 32).to(torch.int32)


def uniform_ints(seed: int, stream: int, n: int, lo: int, hi: int, device="cpu") -> torch.Tensor:
    """n integers uniform in [lo, hi] (inclusive) as int64."""
    h = hash_u32(seed, stream, 0, n, device)
    return lo + ((h * (hi - lo + 1)) >> 32)


def weight_names(shape: ModelShape) -> list[str]:
    """Tensor names, as the checkpoint on the pages names them (lm_head tied to the embedding)."""
    names = ["model.embed_tokens.weight"]
    for i in range(shape.n_layers):
        p = f"model.layers.{i}"
        names += [f"{p}.input_layernorm.weight",
                  f"{p}.self_attn.q_proj.weight", f"{p}.self_attn.k_proj.weight",
                  f"{p}.self_attn.v_proj.weight", f"{p}.self_attn.q_norm.weight",
                  f"{p}.self_attn.k_norm.weight", f"{p}.self_attn.o_proj.weight",
                  f"{p}.post_attention_layernorm.weight",
                  f"{p}.mlp.gate_proj.weight", f"{p}.mlp.up_proj.weight", f"{p}.mlp.down_proj.weight"]
    names.append("model.norm.weight")
    return names


def weight_shapes(shape: ModelShape) -> dict[str, tuple[int, ...]]:
    D, Hq, Hkv, d, I = shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.intermediate
    out = {"model.embed_tokens.weight": (shape.vocab, D), "model.norm.weight": (D,)}
    for i in range(shape.n_layers):
        p = f"model.layers.{i}"
        out.update({
            f"{p}.input_layernorm.weight": (D,),
            f"{p}.self_attn.q_proj.weight": (Hq * d, D),
            f"{p}.self_attn.k_proj.weight": (Hkv * d, D),
            f"{p}.self_attn.v_proj.weight": (Hkv * d, D),
            f"{p}.self_attn.q_norm.weight": (d,),
            f"{p}.self_attn.k_norm.weight": (d,),
            f"{p}.self_attn.o_proj.weight": (D, Hq * d),
            f"{p}.post_attention_layernorm.weight": (D,),
            f"{p}.mlp.gate_proj.weight": (I, D),
            f"{p}.mlp.up_proj.weight": (I, D),
            f"{p}.mlp.down_proj.weight": (D, I),
        })
    return out


def _stream_of(name: str) -> int | None:
    if name == "model.embed_tokens.weight":
        return STREAM_EMBED
    parts = name.split(".")
    if parts[1] == "layers":
        slot = LAYER_SLOTS.get(parts[4]) if len(parts) > 4 else None
        if slot is None:
            return None
        return STREAM_LAYER_BASE + 16 * int(parts[2]) + slot
    return None


def make_weights(shape: ModelShape = QWEN3_0_6B, seed: int = 0, device="cpu") -> dict[str, torch.Tensor]:
    """Random-init bf16 weights: matrices ~N(0, weight_std), norm weights exactly 1.0."""
    w = {}
    for name, shp in weight_shapes(shape).items():
        n = math.prod(shp)
        stream = _stream_of(name)
        if stream is None:
            w[name] = ones_bf16(n, device).view(shp)
        else:
            w[name] = normal_bf16(seed, stream, n, shape.weight_std, device).view(shp)
    return w


def kv_values(seed: int, layer: int, which: int, start: int, n: int, std: float, device="cpu") -> torch.Tensor:
    """Synthetic cache entries (bf16) for one layer; which=0 for K, 1 for V.

    Counter = flat index into a [token, kv_head, head_dim] array of that layer, so a
    caller can generate any sub-range of a sequence's cache independently.
    """
    return normal_bf16(seed, STREAM_KV + 2 * layer + which, n, std, device, start=start)


def bf16_to_f32(t: torch.Tensor) -> torch.Tensor:
    """Exact widening of bf16 bit patterns."""
    return t.view(torch.int16).to(torch.int32).bitwise_left_shift(16).view(torch.float32)
