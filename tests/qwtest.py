"""Helpers for the GPU parity tests: block tables, cache injection, oracle runs
and the comparison rules (relative L2 per row, margin-gated token equality)."""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth

PAGE = 16
SEQ_STRIDE = 1 << 15          # counter stride between sequences in the synthetic caches
K_STD, V_STD = 1.0, 0.64      # keys after QK-Norm have unit RMS; v = h Wv^T with h of unit RMS

# a small model the kernels accept (head_dim 128, Hq = 2 Hkv), for fast end-to-end checks
SMALL = synth.ModelShape(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=128, intermediate=384,
                         vocab=4096, weight_std=0.02)
FULL = synth.QWEN3_0_6B

HIDDEN_TOL = 1e-2
LOGIT_TOL = 1e-2
MARGIN = 0.05


def rel_l2_rows(got, ref) -> np.ndarray:
    got = np.asarray(got, dtype=np.float64).reshape(len(ref), -1)
    ref = np.asarray(ref, dtype=np.float64).reshape(len(ref), -1)
    return np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)


def block_tables(lengths, capacity_tokens, n_pages, seed=0, shuffle=True):
    """One row per sequence with room for capacity_tokens; pages handed out in a
    shuffled order so that the page indirection is exercised.  Returns (int32 table, list of page lists)."""
    per = math.ceil(capacity_tokens / PAGE)
    need = per * len(lengths)
    assert need <= n_pages
    ids = np.arange(n_pages)
    if shuffle:
        ids = np.random.default_rng(seed).permutation(n_pages)
    bt = ids[:need].reshape(len(lengths), per).astype(np.int32)
    return bt, [list(map(int, row)) for row in bt]


def synth_kv(seq: int, layer: int, L: int, n_kv: int, device="cpu"):
    """Synthetic post-RoPE keys and values of one sequence and layer: bf16 [L, n_kv, 128] each."""
    per_tok = n_kv * 128
    start = seq * SEQ_STRIDE * per_tok
    k = synth.kv_values(0, layer, 0, start, L * per_tok, K_STD, device).view(L, n_kv, 128)
    v = synth.kv_values(0, layer, 1, start, L * per_tok, V_STD, device).view(L, n_kv, 128)
    return k, v


def inject(pool: torch.Tensor, layer: int, pages: list[int], k: torch.Tensor, v: torch.Tensor):
    """Write a sequence's [L, n_kv, 128] keys/values into its pages of the pool view."""
    L, n_kv, d = k.shape
    n_p = math.ceil(L / PAGE)
    pad = n_p * PAGE - L
    idx = torch.tensor(pages[:n_p], device=pool.device, dtype=torch.long)
    for which, t in ((0, k), (1, v)):
        t = t.to(pool.device)
        if pad:
            t = torch.cat([t, torch.zeros(pad, n_kv, d, dtype=t.dtype, device=t.device)])
        pool[layer, idx, which] = t.view(n_p, PAGE, n_kv, d).permute(0, 2, 1, 3)


def read_kv(pool: torch.Tensor, layer: int, pages: list[int], L: int):
    """Inverse of inject: ([L, n_kv, 128] K, V) of one sequence from the pool view, as float64 numpy."""
    n_p = math.ceil(L / PAGE)
    idx = torch.tensor(pages[:n_p], device=pool.device, dtype=torch.long)
    out = []
    for which in (0, 1):
        t = pool[layer, idx, which].permute(0, 2, 1, 3).reshape(n_p * PAGE, pool.shape[3], 128)[:L]
        out.append(t.float().cpu().double().numpy())
    return out


def oracle_prefix_cache(shape, seq: int, L: int):
    """Oracle cache holding the synthetic prefix (positions 0..L-1) of one sequence."""
    cache = []
    for layer in range(shape.n_layers):
        k, v = synth_kv(seq, layer, L, shape.n_kv_heads)
        kk = R.bf16_to_f64(k).transpose(1, 0, 2)
        vv = R.bf16_to_f64(v).transpose(1, 0, 2)
        cache.append(R.LayerCache(kk, vv, np.arange(L)))
    return cache


class LazyPrefixCache(list):
    """Oracle cache for one decode step over a long synthetic prefix: each layer's
    prefix is generated when the oracle reaches that layer and dropped afterwards;
    only the newest position of every layer is kept (for checking the cache write)."""

    def __init__(self, shape, seq: int, L: int):
        def make(layer):
            k, v = synth_kv(seq, layer, L, shape.n_kv_heads)
            return R.LayerCache(R.bf16_to_f64(k).transpose(1, 0, 2), R.bf16_to_f64(v).transpose(1, 0, 2),
                                np.arange(L))
        super().__init__([make] * shape.n_layers)

    def __setitem__(self, i, c):
        super().__setitem__(i, R.LayerCache(c.k[:, -1:], c.v[:, -1:], c.pos[-1:]))


def lazy_prefix_cache(shape, seq: int, L: int):
    return LazyPrefixCache(shape, seq, L)


def assert_tokens_match(gpu_ids, ref_logits_rows, ref_ids, margin=MARGIN):
    """Greedy ids must agree wherever the oracle's top-1 / top-2 margin exceeds `margin`."""
    checked = 0
    for i, (g, row, r) in enumerate(zip(gpu_ids, ref_logits_rows, ref_ids)):
        top2 = np.partition(row, -2)[-2:]
        if top2[1] - top2[0] > margin:
            assert int(g) == int(r), f"row {i}: gpu {g} vs oracle {r} (margin {top2[1] - top2[0]:.3f})"
            checked += 1
    return checked


def sample_exempt(detail: dict, top_p: float, tol=1e-3) -> bool:
    """Near-ties the sampling comparison exempts: the draw lands within tol of a cumulative
    boundary of the kept list, or the top-p cutoff sits within tol of top_p."""
    if detail.get("cutoff") is None:
        return False
    return (detail["draw_gap"] < tol or abs(detail["cum_before_cutoff"] - top_p) < tol
            or abs(detail["cum_at_cutoff"] - top_p) < tol)


def split_rows(a: torch.Tensor) -> torch.Tensor:
    """The hi/lo bf16 layout of float rows a[M][K] that split-mode projections read."""
    M, K = a.shape
    tiles = (M + 63) // 64
    out = torch.zeros(tiles * 128, K, dtype=torch.bfloat16, device=a.device)
    hi = a.to(torch.bfloat16)
    lo = (a - hi.float()).to(torch.bfloat16)
    idx = torch.arange(M, device=a.device)
    dst = (idx // 64) * 128 + idx % 64
    out[dst] = hi
    out[dst + 64] = lo
    return out


def sample_draw_is_valid(logits, temperature: float, top_k: int, top_p: float, u: float, got: int,
                         eps: float = 2e-4) -> bool:
    """Whether `got` is the inverse-CDF draw of u from Step 8's kept list up to rounding of the
    cumulative sums: its rank in (probability desc, id asc) order lies in the top-p prefix (and
    under top_k), and its cumulative interval, normalised by the kept mass, contains u within
    eps.  Used where the exact comparison is exempt (large nuclei: boundaries closer than 1e-3)."""
    z = np.asarray(logits, dtype=np.float64) / temperature
    p = np.exp(z - z.max())
    p /= p.sum()
    order = np.lexsort((np.arange(p.size), -p))
    c = np.cumsum(p[order])
    cutoff = int(np.sum(c < top_p)) + 1
    if top_k > 0:
        cutoff = min(cutoff, top_k)
    cutoff = min(cutoff, p.size)
    kept_mass = c[cutoff - 1]
    rank = int(np.nonzero(order == got)[0][0])
    c_prev = c[rank - 1] if rank else 0.0
    in_prefix = rank < cutoff or c_prev < top_p + eps
    under_k = top_k <= 0 or rank < top_k
    in_interval = c_prev / kept_mass <= u + eps and c[rank] / kept_mass >= u - eps
    return in_prefix and under_k and in_interval


def c_oracle_prefix_cache(corc, shape, seq: int, L: int, extra: int = 1):
    """The C oracle's cache of one sequence holding the synthetic prefix (positions 0..L-1),
    with room for `extra` more positions; values from the seeded generator (run on the GPU when
    there is one: it is bit-identical on every device)."""
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    cache = corc.new_cache(L + extra)
    for layer in range(shape.n_layers):
        k, v = synth_kv(seq, layer, L, shape.n_kv_heads, device=dev)
        cache.fill_prefix(layer, k.float().cpu().numpy(), v.float().cpu().numpy())
    cache.set_len(L)
    return cache
