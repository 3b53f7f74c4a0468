"""Plain CPU oracle of the Qwen3-0.6B decoder forward pass, KV cache and sampler.

TEST INFRASTRUCTURE ONLY (see the package docstring): never on the product path.

Source: the article "Inside an LLM: Pure Python Inference for Qwen3-0.6B on MLX"
(English page), steps 2-9.  Each function names the step it restates.

Precision
  * float64 everywhere; bf16 weights are widened exactly.
  * RoPE (Step 4) is the one place the article fixes a precision: its inverse
    frequencies and angles are float32 arrays.  The oracle keeps both in float32
    (inv_freq_i = float32(theta^(-i/half)), angle = float32(float32(pos) * inv_freq_i))
    and evaluates cos/sin in float64 on those float32 angles.

Readings of points the article leaves open
  * forward(ids, cache, pos) is called in Step 9 but never shown: embedding
    (Step 2) -> n_layers x transformer_block (Step 7) -> final RMSNorm + LM head
    (Step 8), the only order consistent with the steps.
  * The causal mask of Step 5 (triu of -1e9 when seq_len > 1) is read as
    "key j is visible to a query iff position(j) <= position(query)"; it equals the
    article's mask whenever the cache starts empty and excludes keys exactly
    (exp(-1e9 - max) is 0 in float64 anyway).
  * The LM head is tied to the embedding matrix (model.embed_tokens.weight).
  * sample() (Step 8): top-k is applied as a cap on the article's top-p cutoff,
    ties in the descending sort go to the lower token id, and the categorical draw
    is an inverse-CDF draw on the kept, renormalised list with u in [0, 1).
"""
from __future__ import annotations

import numpy as np
import torch

EPS = 1e-6          # Step 3, RMSNorm
THETA = 1e6         # Step 4, RoPE base frequency for Qwen3
M32 = 0xFFFFFFFF


def bf16_to_f64(t) -> np.ndarray:
    """Exact widening of bf16 values (torch.bfloat16 tensor or uint16 bit array) to float64."""
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").contiguous().view(torch.bfloat16).to(torch.float64).numpy()
    bits = np.asarray(t, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even to bf16, returned as float64 (used only for error attribution)."""
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) & 0xFFFF
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- Step 3: RMSNorm
def rms_norm(x: np.ndarray, w: np.ndarray, eps: float = EPS) -> np.ndarray:
    """x / sqrt(mean(x^2 over the last axis) + eps) * w (no mean subtraction, no bias)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


# ---------------------------------------------------------------- Step 4: RoPE
def rope_inv_freq(head_dim: int, theta: float = THETA) -> np.ndarray:
    """float32 inverse frequencies theta^(-i/half), i = 0 .. half-1 (half = head_dim/2)."""
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    return (1.0 / np.power(theta, i / half)).astype(np.float32)


def rope_angles(positions, head_dim: int, theta: float = THETA) -> np.ndarray:
    """float32 angle table [T, half]: float32(position) * inv_freq, rounded to float32."""
    pos = np.asarray(positions, dtype=np.float32)
    return pos[:, None] * rope_inv_freq(head_dim, theta)[None, :]


def apply_rope(x: np.ndarray, positions, theta: float = THETA) -> np.ndarray:
    """Half-split rotation of x[..., T, head_dim]: pair (i, i + half) turns by angle[t, i]."""
    d = x.shape[-1]
    half = d // 2
    ang = rope_angles(positions, d, theta).astype(np.float64)
    cos, sin = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x1 * sin + x2 * cos], axis=-1)


# ---------------------------------------------------------------- Step 6: SwiGLU
def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g * sigmoid(g)."""
    return g / (1.0 + np.exp(-g))


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def gqa_attention(q, k, v, kpos, qpos):
    """Step 5 core: softmax(q k^T / sqrt(d)) v per query head, query head h reading kv
    head h // (n_heads / n_kv_heads) (the article expands K and V with repeat), keys at
    positions above the query's position excluded.

    q [Hq, T, d], k and v [Hkv, L, d], kpos [L], qpos [T] -> [Hq, T, d]."""
    Hq, T, d = q.shape
    group = Hq // k.shape[0]
    K = np.repeat(k, group, axis=0)
    V = np.repeat(v, group, axis=0)
    visible = np.asarray(kpos, dtype=np.int64)[None, :] <= np.asarray(qpos, dtype=np.int64)[:, None]
    out = np.empty((Hq, T, d))
    for h in range(Hq):
        scores = (q[h] @ K[h].T) * d ** -0.5
        scores = np.where(visible, scores, -np.inf)
        out[h] = softmax(scores) @ V[h]
    return out


class LayerCache:
    """Per-layer, per-sequence cache of post-RoPE keys and values (Step 5, 'The KV cache').

    k, v: [n_kv_heads, L, head_dim] float64; pos: [L] positions of the cached keys.
    """
    def __init__(self, k, v, pos):
        self.k, self.v, self.pos = k, v, np.asarray(pos, dtype=np.int64)

    def append(self, k, v, pos):
        self.k = np.concatenate([self.k, k], axis=1)
        self.v = np.concatenate([self.v, v], axis=1)
        self.pos = np.concatenate([self.pos, np.asarray(pos, dtype=np.int64)])


# ---------------------------------------------------------------- weight-only int8 (not in the article)
# The article's "What the script leaves out" section names quantisation without defining one.
# Reading used here: symmetric int8 per output channel (per row of an [out][in] matrix, and per
# vocabulary row of the tied embedding / LM head) with a power-of-two scale:
#   t_r = float32(max_c |w_rc|) / 127 (IEEE float32 division),
#   scale_r = the smallest power of two >= t_r,
#   q_rc = round_half_even(w_rc / scale_r) (exact: a division by a power of two), in [-127, 127];
# a row of zeros has scale 0 and codes 0.  The model computes with q_rc * scale_r, which (seven
# magnitude bits times a power of two) is exactly representable in bf16, so a path that streams
# the codes and a path that streams bf16 compute with the same weights.
QUANTISED_SUFFIXES = ("q_proj.weight", "k_proj.weight", "v_proj.weight", "o_proj.weight",
                      "gate_proj.weight", "up_proj.weight", "down_proj.weight")


def pow2_ceil(t: np.ndarray) -> np.ndarray:
    """Smallest power of two >= t for positive float32 t (0 stays 0), as float32."""
    t = np.asarray(t, np.float32)
    m, e = np.frexp(t)                       # t = m * 2^e, m in [0.5, 1)
    s = np.ldexp(np.float32(1), np.where(m == 0.5, e - 1, e)).astype(np.float32)
    return np.where(t > 0, s, np.float32(0)).astype(np.float32)


def quantize_rows_int8(w) -> tuple[np.ndarray, np.ndarray]:
    """Per-row symmetric int8 codes and power-of-two float32 scales of a [rows][cols] matrix."""
    w32 = bf16_to_f64(w).astype(np.float32) if isinstance(w, torch.Tensor) else np.asarray(w, np.float32)
    amax = np.max(np.abs(w32), axis=1).astype(np.float32)
    scale = pow2_ceil((amax / np.float32(127)).astype(np.float32))
    safe = np.where(scale > 0, scale, np.float32(1)).astype(np.float32)
    q = np.rint((w32 / safe[:, None]).astype(np.float32))
    q = np.where(scale[:, None] > 0, np.clip(q, -127, 127), 0).astype(np.int8)
    return q, scale


def dequantize_rows_int8(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """The weights the quantised model computes with: q_rc * scale_r, in float64."""
    return q.astype(np.float64) * scale.astype(np.float64)[:, None]


class Qwen3Oracle:
    """The model of steps 2-8 over one sequence at a time, weights as float64 numpy arrays.

    weight_bits = 8: the projection matrices and the tied embedding are replaced by their
    dequantised per-row int8 values (quantize_rows_int8); norm weights are kept."""

    def __init__(self, weights: dict, shape, eps: float = EPS, theta: float = THETA,
                 kv_round_bf16: bool = False, weight_bits: int = 16):
        self.shape = shape
        self.eps, self.theta = eps, theta
        self.kv_round_bf16 = kv_round_bf16
        self.W = {name: bf16_to_f64(t) for name, t in weights.items()}
        if weight_bits == 8:
            for name in self.W:
                if name == "model.embed_tokens.weight" or name.endswith(QUANTISED_SUFFIXES):
                    self.W[name] = dequantize_rows_int8(*quantize_rows_int8(self.W[name]))
        elif weight_bits != 16:
            raise ValueError("weight_bits must be 16 or 8")

    # Step 5: attention with grouped query heads
    def attention(self, x, layer, cache, positions):
        S = self.shape
        W = self.W
        p = f"model.layers.{layer}.self_attn"
        T = x.shape[0]
        q = x @ W[f"{p}.q_proj.weight"].T
        k = x @ W[f"{p}.k_proj.weight"].T
        v = x @ W[f"{p}.v_proj.weight"].T
        q = q.reshape(T, S.n_heads, S.head_dim).transpose(1, 0, 2)
        k = k.reshape(T, S.n_kv_heads, S.head_dim).transpose(1, 0, 2)
        v = v.reshape(T, S.n_kv_heads, S.head_dim).transpose(1, 0, 2)
        q = rms_norm(q, W[f"{p}.q_norm.weight"], self.eps)          # QK-Norm before RoPE
        k = rms_norm(k, W[f"{p}.k_norm.weight"], self.eps)
        q = apply_rope(q, positions, self.theta)
        k = apply_rope(k, positions, self.theta)
        if self.kv_round_bf16:
            k, v = round_to_bf16(k), round_to_bf16(v)
        c = cache[layer]
        if callable(c):                       # a lazily generated cache prefix
            c = c(layer)
        if c is None:
            c = LayerCache(k, v, positions)
        else:
            c.append(k, v, positions)
        cache[layer] = c
        out = gqa_attention(q, c.k, c.v, c.pos, positions)
        out = out.transpose(1, 0, 2).reshape(T, S.n_heads * S.head_dim)
        return out @ W[f"{p}.o_proj.weight"].T

    # Step 6: SwiGLU feed-forward
    def ffn(self, x, layer):
        W = self.W
        p = f"model.layers.{layer}.mlp"
        gate = x @ W[f"{p}.gate_proj.weight"].T
        up = x @ W[f"{p}.up_proj.weight"].T
        return (silu(gate) * up) @ W[f"{p}.down_proj.weight"].T

    # Step 7: pre-norm block with residuals
    def transformer_block(self, x, layer, cache, positions):
        p = f"model.layers.{layer}"
        h = rms_norm(x, self.W[f"{p}.input_layernorm.weight"], self.eps)
        x = x + self.attention(h, layer, cache, positions)
        h = rms_norm(x, self.W[f"{p}.post_attention_layernorm.weight"], self.eps)
        x = x + self.ffn(h, layer)
        return x

    def new_cache(self):
        return [None] * self.shape.n_layers

    # Step 2 + Step 7 x n_layers + Step 8 (final norm and tied LM head)
    def forward(self, ids, positions, cache, last_only: bool = False, hiddens: list | None = None,
                vocab_chunk: int = 16384):
        """Logits [T, vocab] (or [1, vocab] with last_only) for one sequence's tokens."""
        ids = np.asarray(ids, dtype=np.int64)
        positions = np.asarray(positions, dtype=np.int64)
        E = self.W["model.embed_tokens.weight"]
        x = E[ids]
        for layer in range(self.shape.n_layers):
            x = self.transformer_block(x, layer, cache, positions)
            if hiddens is not None:
                hiddens.append(x.copy())
        if last_only:
            x = x[-1:]
        return self.lm_head(x, vocab_chunk)

    def lm_head(self, x, vocab_chunk: int = 16384):
        E = self.W["model.embed_tokens.weight"]
        h = rms_norm(x, self.W["model.norm.weight"], self.eps)
        out = np.empty((h.shape[0], E.shape[0]))
        for v0 in range(0, E.shape[0], vocab_chunk):
            out[:, v0:v0 + vocab_chunk] = h @ E[v0:v0 + vocab_chunk].T
        return out


# ---------------------------------------------------------------- Step 8: sampling
def sample(logits, temperature: float, top_k: int, top_p: float, u: float) -> int:
    return sample_detail(logits, temperature, top_k, top_p, u)["id"]


def sample_detail(logits, temperature: float, top_k: int, top_p: float, u: float) -> dict:
    """sample() of Step 8 with a top-k cap and an explicit uniform draw u in [0, 1).

    Greedy (argmax, lowest id on ties) when temperature == 0.  Otherwise
    p = softmax(logits / T) over the whole vocabulary, sorted descending,
    cutoff = #(cumsum < top_p) + 1, capped at top_k (top_k <= 0: no cap),
    kept probabilities renormalised, and the first j with cumsum(kept)_j > u
    is returned.  The dict also carries the quantities the parity tests need
    to recognise near-ties.
    """
    logits = np.asarray(logits, dtype=np.float64)
    srt = np.sort(logits)[::-1]
    margin = float(srt[0] - srt[1]) if logits.size > 1 else float("inf")
    if temperature == 0:
        return {"id": int(np.argmax(logits)), "margin": margin}
    p = softmax(logits / temperature)
    order = np.argsort(-p, kind="stable")
    sp = p[order]
    c = np.cumsum(sp)
    cutoff = int(np.sum(c < top_p)) + 1
    if top_k > 0:
        cutoff = min(cutoff, top_k)
    cutoff = min(cutoff, sp.size)
    kept = sp[:cutoff] / np.sum(sp[:cutoff])
    ck = np.cumsum(kept)
    j = int(np.searchsorted(ck, u, side="right"))   # first j with ck[j] > u
    j = min(j, cutoff - 1)
    return {"id": int(order[j]), "margin": margin, "cutoff": cutoff, "kept": order[:cutoff],
            "cum_at_cutoff": float(c[cutoff - 1]), "cum_before_cutoff": float(c[cutoff - 2]) if cutoff > 1 else 0.0,
            "draw_gap": float(np.min(np.abs(ck - u))), "u": u}


# ------------------------------------------- counter-based RNG for the draw
# Philox4x32-10 of Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy
# as 1, 2, 3" (SC'11): ten rounds of two 32x32->64 multiplies on a 4-word counter,
# with a Weyl-sequence key schedule.
PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85


def philox4x32_10(ctr, key):
    c0, c1, c2, c3 = (int(v) & M32 for v in ctr)
    k0, k1 = (int(v) & M32 for v in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + PHILOX_W0) & M32
            k1 = (k1 + PHILOX_W1) & M32
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & M32, p1 & M32, ((p0 >> 32) ^ c3 ^ k1) & M32, p0 & M32
    return c0, c1, c2, c3


def sampling_uniform(seed: int, rng_counter: int) -> float:
    """The draw for one sequence at one step: key = 64-bit seed, counter = (rng_counter, 0, 0);
    u = (first output word >> 8) * 2^-24, exactly representable in float32."""
    r = philox4x32_10((rng_counter & M32, (rng_counter >> 32) & M32, 0, 0), (seed & M32, (seed >> 32) & M32))
    return (r[0] >> 8) * 2.0 ** -24


# ---------------------------------------------------------------- Step 9: generation loop
def generate(model: Qwen3Oracle, prompt_ids, n_steps: int, temperature: float = 0.0, top_k: int = 0,
             top_p: float = 1.0, seed: int = 0, forced=None):
    """Prefill once, then decode one token at a time (no EOS: fixed step count).

    Returns (chosen ids, per-step logits rows).  With `forced`, the token fed at
    decode step i is forced[i] instead of the sampled one (teacher forcing).
    """
    cache = model.new_cache()
    T = len(prompt_ids)
    logits = model.forward(prompt_ids, np.arange(T), cache, last_only=True)
    rows = [logits[0]]
    chosen = [sample(logits[0], temperature, top_k, top_p, sampling_uniform(seed, 0))]
    for i in range(1, n_steps):
        nxt = chosen[-1] if forced is None else forced[i - 1]
        pos = T + i - 1
        logits = model.forward([nxt], [pos], cache, last_only=True)
        rows.append(logits[0])
        chosen.append(sample(logits[0], temperature, top_k, top_p, sampling_uniform(seed, i)))
    return chosen, rows
