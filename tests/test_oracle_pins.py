"""Pins of the CPU oracle to facts other than itself (closed forms, invariants,
brute force on tiny inputs, published known-answer vectors).  CPU only."""
import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest

from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ RMSNorm (Step 3)
def test_rmsnorm_unit_rms_when_weight_is_one():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 1024)) * np.array([[1e-1], [1.0], [7.0], [30.0], [1e3]])
    y = R.rms_norm(x, np.ones(1024))
    ms = np.mean(x * x, axis=-1)
    # output RMS is sqrt(ms / (ms + eps)): 1 when ms >> eps, slightly less otherwise
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), np.sqrt(ms / (ms + 1e-6)), rtol=1e-12)
    np.testing.assert_allclose(np.sqrt(np.mean(y[1:] ** 2, axis=-1)), 1.0, rtol=1e-6)


def test_rmsnorm_scale_invariance_and_per_feature_weight():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(3, 128))
    w = rng.normal(size=128)
    for c in (0.5, 3.0, 100.0):
        np.testing.assert_allclose(R.rms_norm(c * x, w), R.rms_norm(x, w), rtol=1e-5, atol=1e-9)
    np.testing.assert_allclose(R.rms_norm(x, w), w * R.rms_norm(x, np.ones(128)), rtol=1e-14)


def test_rmsnorm_worked_values_and_eps_inside_sqrt():
    # [3, 4]: mean square 12.5 -> [3, 4] / 3.5355339... (eps negligible)
    y = R.rms_norm(np.array([3.0, 4.0]), np.ones(2))
    np.testing.assert_allclose(y, [0.8485281374238570, 1.1313708498984760], rtol=1e-6)
    # mean square equal to eps: the factor is 1/sqrt(2 eps), so 1e-3 -> 1/sqrt(2)
    y = R.rms_norm(np.full(8, 1e-3), np.ones(8))
    np.testing.assert_allclose(y, 1 / math.sqrt(2), rtol=1e-12)
    assert np.all(R.rms_norm(np.zeros(4), np.ones(4)) == 0.0)       # no division by zero


# ------------------------------------------------------------------ RoPE (Step 4)
def test_rope_inverse_frequency_endpoints():
    f = R.rope_inv_freq(128, 1e6)
    assert f.dtype == np.float32 and f.shape == (64,)
    assert f[0] == 1.0                                            # 1 radian per position
    np.testing.assert_allclose(f[63], 10.0 ** (-6 * 63 / 64), rtol=1e-7)
    np.testing.assert_allclose(f[32], 1e-3, rtol=1e-7)            # theta^(-1/2)
    assert np.all(np.diff(f) < 0)


def test_rope_position_zero_is_identity_and_norms_are_kept():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(2, 5, 128))
    np.testing.assert_array_equal(R.apply_rope(x[:, :1], [0]), x[:, :1])
    y = R.apply_rope(x, [0, 1, 7, 300, 32799])
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    # each (i, i+64) pair keeps its own length
    np.testing.assert_allclose(np.hypot(y[..., :64], y[..., 64:]), np.hypot(x[..., :64], x[..., 64:]), rtol=1e-12)


def test_rope_half_split_basis_vectors():
    """e_i turns into cos at i and sin at i+half; e_{i+half} into -sin at i and cos at i+half."""
    d, half, pos = 128, 64, 3
    for i in (0, 5, 63):
        f = 10.0 ** (-6 * i / 64)                     # theta^(-i/64), theta = 1e6
        e = np.zeros((1, d)); e[0, i] = 1.0
        y = R.apply_rope(e, [pos])[0]
        np.testing.assert_allclose([y[i], y[i + half]], [math.cos(pos * f), math.sin(pos * f)], atol=1e-6)
        assert np.count_nonzero(np.abs(y) > 1e-12) <= 2
        e = np.zeros((1, d)); e[0, i + half] = 1.0
        y = R.apply_rope(e, [pos])[0]
        np.testing.assert_allclose([y[i], y[i + half]], [-math.sin(pos * f), math.cos(pos * f)], atol=1e-6)


def test_rope_scores_depend_only_on_distance():
    rng = np.random.default_rng(4)
    q = rng.normal(size=(1, 128))
    k = rng.normal(size=(1, 128))
    for m, n, s in [(3, 1, 5), (10, 2, 17), (0, 9, 40)]:
        a = R.apply_rope(q, [m])[0] @ R.apply_rope(k, [n])[0]
        b = R.apply_rope(q, [m + s])[0] @ R.apply_rope(k, [n + s])[0]
        assert abs(a - b) < 1e-4 * (1 + abs(a))


# ------------------------------------------------------------------ SwiGLU (Step 6)
def test_silu_special_values():
    assert R.silu(np.array(0.0)) == 0.0
    np.testing.assert_allclose(R.silu(np.array(1.0)), 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    np.testing.assert_allclose(R.silu(np.array(30.0)), 30.0, rtol=1e-12)
    assert abs(R.silu(np.array(-30.0))) < 1e-11


# ------------------------------------------------------------------ tiny model helpers
def _tiny_model(shape, seed=0, **kw):
    w = synth.make_weights(shape, seed=seed)
    return w, R.Qwen3Oracle(w, shape, **kw)


def _brute_attention(h, Wq, Wk, Wv, qn, kn, positions, past, n_heads, n_kv, d):
    """Scalar-loop attention of one layer (no o_proj): returns rows [T][n_heads*d] and appends to past."""
    def rms(vec, w):
        ms = sum(t * t for t in vec) / len(vec)
        return [t / math.sqrt(ms + R.EPS) * wi for t, wi in zip(vec, w)]

    def mat_vec(W, x):
        return [sum(W[r][c] * x[c] for c in range(len(x))) for r in range(len(W))]

    def rope(vec, p):
        half = len(vec) // 2
        out = [0.0] * len(vec)
        for i in range(half):
            f = float(np.float32(1.0 / (1e6 ** (i / half))))
            a = float(np.float32(np.float32(p) * np.float32(f)))
            out[i] = vec[i] * math.cos(a) - vec[i + half] * math.sin(a)
            out[i + half] = vec[i] * math.sin(a) + vec[i + half] * math.cos(a)
        return out

    rows = []
    for t, p in enumerate(positions):
        q, k, v = mat_vec(Wq, h[t]), mat_vec(Wk, h[t]), mat_vec(Wv, h[t])
        qh = [rope(rms(q[j * d:(j + 1) * d], qn), p) for j in range(n_heads)]
        kh = [rope(rms(k[j * d:(j + 1) * d], kn), p) for j in range(n_kv)]
        vh = [v[j * d:(j + 1) * d] for j in range(n_kv)]
        past.append((p, kh, vh))
        row = []
        for j in range(n_heads):
            g = j // (n_heads // n_kv)
            vis = [(kp, kk[g], vv[g]) for kp, kk, vv in past if kp <= p]
            s = [sum(a * b for a, b in zip(qh[j], kk)) / math.sqrt(d) for _, kk, _ in vis]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            z = sum(e)
            row += [sum(e[i] * vis[i][2][c] for i in range(len(vis))) / z for c in range(d)]
        rows.append(row)
    return rows


def test_attention_matches_scalar_brute_force_with_cache(tiny_shape):
    S = tiny_shape
    w, m = _tiny_model(S)
    Wo = m.W["model.layers.0.self_attn.o_proj.weight"]
    m.W["model.layers.0.self_attn.o_proj.weight"] = np.eye(S.hidden)   # expose the merged heads
    rng = np.random.default_rng(5)
    p = "model.layers.0.self_attn"
    args = [m.W[f"{p}.{n}.weight"].tolist() for n in ("q_proj", "k_proj", "v_proj")]
    args += [m.W[f"{p}.q_norm.weight"].tolist(), m.W[f"{p}.k_norm.weight"].tolist()]
    cache, past = m.new_cache(), []
    for chunk in ([0, 1, 2, 3, 4], [5], [6, 7]):                  # prefill, decode, chunk
        h = rng.normal(size=(len(chunk), S.hidden))
        got = m.attention(h, 0, cache, chunk)
        ref = _brute_attention(h.tolist(), *args, chunk, past, S.n_heads, S.n_kv_heads, S.head_dim)
        np.testing.assert_allclose(got, np.array(ref), rtol=1e-10, atol=1e-12)
    m.W["model.layers.0.self_attn.o_proj.weight"] = Wo


def test_attention_identical_keys_average_visible_values(tiny_shape):
    S = tiny_shape
    _, m = _tiny_model(S)
    p = "model.layers.0.self_attn"
    m.W[f"{p}.k_proj.weight"] = np.zeros_like(m.W[f"{p}.k_proj.weight"])   # every key is 0 -> equal scores
    m.W[f"{p}.o_proj.weight"] = np.eye(S.hidden)
    h = np.random.default_rng(6).normal(size=(4, S.hidden))
    out = m.attention(h, 0, m.new_cache(), [0, 1, 2, 3])
    v = (h @ m.W[f"{p}.v_proj.weight"].T).reshape(4, S.n_kv_heads, S.head_dim)
    group = S.n_heads // S.n_kv_heads
    for t in range(4):
        for j in range(S.n_heads):
            expect = v[: t + 1, j // group].mean(axis=0)
            np.testing.assert_allclose(out[t, j * S.head_dim:(j + 1) * S.head_dim], expect, rtol=1e-12)
    # a single visible key returns its value exactly
    np.testing.assert_allclose(out[0, :S.head_dim], v[0, 0], rtol=1e-12)


def test_gqa_query_head_uses_kv_head_h_div_group(tiny_shape):
    S = tiny_shape
    _, m = _tiny_model(S)
    p = "model.layers.0.self_attn"
    Wv = m.W[f"{p}.v_proj.weight"].copy()
    Wv[: S.head_dim] = 0.0                              # kv head 0 carries zero values
    m.W[f"{p}.v_proj.weight"] = Wv
    m.W[f"{p}.o_proj.weight"] = np.eye(S.hidden)
    out = m.attention(np.random.default_rng(7).normal(size=(3, S.hidden)), 0, m.new_cache(), [0, 1, 2])
    per_head = np.abs(out).reshape(3, S.n_heads, S.head_dim).sum(axis=(0, 2))
    group = S.n_heads // S.n_kv_heads
    for j in range(S.n_heads):
        assert (per_head[j] == 0.0) == (j // group == 0)


def test_causality_future_tokens_do_not_change_earlier_rows(tiny_shape):
    _, m = _tiny_model(tiny_shape)
    a = m.forward([5, 9, 100, 3, 7], np.arange(5), m.new_cache())
    b = m.forward([5, 9, 100, 250, 1], np.arange(5), m.new_cache())
    np.testing.assert_array_equal(a[:3], b[:3])
    assert np.abs(a[3:] - b[3:]).max() > 1e-3


def test_cached_decode_equals_full_recompute(tiny_shape):
    _, m = _tiny_model(tiny_shape)
    ids = [11, 200, 3, 3, 42, 255, 0, 17]
    full = m.forward(ids, np.arange(len(ids)), m.new_cache())
    cache = m.new_cache()
    rows = [m.forward(ids[:5], np.arange(5), cache)[-1]]
    for t in range(5, len(ids)):
        rows.append(m.forward([ids[t]], [t], cache)[-1])
    np.testing.assert_allclose(np.array(rows), full[4:], rtol=1e-11, atol=1e-12)
    # two prefill chunks equal one prefill of the concatenation
    cache = m.new_cache()
    m.forward(ids[:3], np.arange(3), cache)
    np.testing.assert_allclose(m.forward(ids[3:], np.arange(3, 8), cache), full[3:], rtol=1e-11, atol=1e-12)


def test_zero_projections_leave_embedding_and_tie_the_head(tiny_shape):
    """With every projection zero the blocks add nothing: logits = rms(E[id]) . E[j] (scalar loops)."""
    S = tiny_shape
    _, m = _tiny_model(S)
    for k in list(m.W):
        if k.endswith("proj.weight"):
            m.W[k] = np.zeros_like(m.W[k])
    E = m.W["model.embed_tokens.weight"]
    got = m.forward([7, 123], [0, 1], m.new_cache())
    for r, tok in enumerate([7, 123]):
        e = E[tok].tolist()
        s = 1.0 / math.sqrt(sum(t * t for t in e) / len(e) + R.EPS)
        for j in (0, 1, tok, S.vocab - 1):
            expect = sum(e[c] * s * E[j][c] for c in range(S.hidden))
            assert abs(got[r, j] - expect) < 1e-12 * (1 + abs(expect))


def test_single_token_block_is_x_plus_o_v_of_normed_x(tiny_shape):
    """One visible key: softmax weight 1, so attention(h) = Wo Wv h whatever q and k are."""
    S = tiny_shape
    _, m = _tiny_model(S)
    p = "model.layers.0"
    x = np.random.default_rng(8).normal(size=(1, S.hidden))
    h = R.rms_norm(x, m.W[f"{p}.input_layernorm.weight"])
    got = m.attention(h, 0, m.new_cache(), [9])
    Wv, Wo = m.W[f"{p}.self_attn.v_proj.weight"], m.W[f"{p}.self_attn.o_proj.weight"]
    v = (h @ Wv.T).reshape(S.n_kv_heads, S.head_dim)
    group = S.n_heads // S.n_kv_heads
    merged = np.concatenate([v[j // group] for j in range(S.n_heads)])   # query head j reads kv head j // group
    np.testing.assert_allclose(got[0], Wo @ merged, rtol=1e-11)


def test_ffn_matches_scalar_loops(tiny_shape):
    S = tiny_shape
    _, m = _tiny_model(S)
    p = "model.layers.1.mlp"
    Wg, Wu, Wd = (m.W[f"{p}.{n}.weight"] for n in ("gate_proj", "up_proj", "down_proj"))
    x = np.random.default_rng(9).normal(size=(2, S.hidden))
    got = m.ffn(x, 1)
    for r in range(2):
        a = []
        for i in range(S.intermediate):
            g = sum(Wg[i][c] * x[r][c] for c in range(S.hidden))
            u = sum(Wu[i][c] * x[r][c] for c in range(S.hidden))
            a.append(g / (1 + math.exp(-g)) * u)
        for o in range(S.hidden):
            expect = sum(Wd[o][i] * a[i] for i in range(S.intermediate))
            assert abs(got[r, o] - expect) < 1e-11 * (1 + abs(expect))


def _scalar_ffn(W, prefix, x_row, S):
    a = []
    Wg, Wu, Wd = (W[f"{prefix}.{n}.weight"] for n in ("gate_proj", "up_proj", "down_proj"))
    for i in range(S.intermediate):
        g = sum(Wg[i][c] * x_row[c] for c in range(S.hidden))
        u = sum(Wu[i][c] * x_row[c] for c in range(S.hidden))
        a.append(g / (1 + math.exp(-g)) * u)
    return [sum(Wd[o][i] * a[i] for i in range(S.intermediate)) for o in range(S.hidden)]


def test_transformer_block_matches_scalar_loops(tiny_shape):
    """Step 7 composition with every sublayer active: h = rms(x, w_in); x1 = x + Wo attn(h);
    x2 = x1 + ffn(rms(x1, w_post)).  Distinct random norm weights catch a swapped weight, an
    FFN fed rms(x) instead of rms(x1), or a dropped residual."""
    S = tiny_shape
    _, m = _tiny_model(S)
    rng = np.random.default_rng(12)
    pl = "model.layers.1"
    w_in = 1.0 + 0.5 * rng.normal(size=S.hidden)
    w_post = 1.0 + 0.5 * rng.normal(size=S.hidden)
    m.W[f"{pl}.input_layernorm.weight"], m.W[f"{pl}.post_attention_layernorm.weight"] = w_in, w_post
    pa = f"{pl}.self_attn"
    args = [m.W[f"{pa}.{n}.weight"].tolist() for n in ("q_proj", "k_proj", "v_proj")]
    args += [m.W[f"{pa}.q_norm.weight"].tolist(), m.W[f"{pa}.k_norm.weight"].tolist()]
    Wo = m.W[f"{pa}.o_proj.weight"]

    def rms(vec, w):
        ms = sum(t * t for t in vec) / len(vec)
        return [t / math.sqrt(ms + R.EPS) * wi for t, wi in zip(vec, w)]

    cache, past = m.new_cache(), []
    for chunk in ([0, 1, 2], [3]):                         # prefill, then one cached decode step
        x = rng.normal(size=(len(chunk), S.hidden))
        got = m.transformer_block(x, 1, cache, chunk)
        h = [rms(list(row), w_in) for row in x]
        att = _brute_attention(h, *args, chunk, past, S.n_heads, S.n_kv_heads, S.head_dim)
        for t in range(len(chunk)):
            x1 = [x[t][o] + sum(Wo[o][c] * att[t][c] for c in range(S.n_heads * S.head_dim))
                  for o in range(S.hidden)]
            f = _scalar_ffn(m.W, f"{pl}.mlp", rms(x1, w_post), S)
            expect = [x1[o] + f[o] for o in range(S.hidden)]
            np.testing.assert_allclose(got[t], expect, rtol=1e-10, atol=1e-12)


def test_generate_positions_and_per_step_counter(tiny_shape):
    """Step 9: the token chosen at step i - 1 is decoded at position T + i - 1, so every logits
    row equals the last row of a fresh full recompute over prompt + chosen ids; step i draws
    its uniform with rng_counter = i."""
    _, m = _tiny_model(tiny_shape)
    prompt = [3, 77, 200, 5]
    T = len(prompt)
    for temp, top_k, top_p in ((0.0, 0, 1.0), (1.3, 0, 0.9), (0.8, 5, 1.0)):
        chosen, rows = R.generate(m, prompt, 5, temperature=temp, top_k=top_k, top_p=top_p, seed=9)
        assert len(chosen) == len(rows) == 5
        for i in range(5):
            seq = prompt + chosen[:i]
            ref = m.forward(seq, np.arange(T + i), m.new_cache())[-1]
            np.testing.assert_allclose(rows[i], ref, rtol=1e-10, atol=1e-12)
            assert chosen[i] == R.sample(ref, temp, top_k, top_p, R.sampling_uniform(9, i))
    # a wrong position is visible in the logits: decoding the same token one position later differs
    cache = m.new_cache()
    m.forward(prompt, np.arange(T), cache)
    a = m.forward([chosen[0]], [T], [c for c in cache])[-1]
    cache2 = m.new_cache()
    m.forward(prompt, np.arange(T), cache2)
    b = m.forward([chosen[0]], [T + 1], cache2)[-1]
    assert np.abs(a - b).max() > 1e-6
    # teacher forcing feeds forced[i - 1] at step i
    forced = [9, 8, 7, 6]
    _, rows_f = R.generate(m, prompt, 5, forced=forced)
    np.testing.assert_allclose(rows_f[4], m.forward(prompt + forced, np.arange(T + 4), m.new_cache())[-1],
                               rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------------ sampling (Step 8)
def test_sample_greedy_and_top1():
    rng = np.random.default_rng(10)
    lg = rng.normal(size=1000)
    lg[417] = 9.0
    assert R.sample(lg, 0.0, 0, 0.9, 0.5) == 417
    for u in (0.0, 0.3, 0.999):
        assert R.sample(lg, 0.7, 1, 0.9, u) == 417
    tie = np.zeros(10); tie[[3, 6]] = 1.0
    assert R.sample(tie, 0.0, 0, 1.0, 0.0) == 3                  # lowest id wins a tie


def test_sample_worked_example_cutoff_rule():
    """p = [0.5, 0.2, 0.3]: sorted [0.5, 0.3, 0.2], cumsum [0.5, 0.8, 1.0]."""
    lg = np.log([0.5, 0.2, 0.3])
    d = R.sample_detail(lg, 1.0, 0, 0.79, 0.0)
    assert d["cutoff"] == 2 and list(d["kept"]) == [0, 2]      # #(c < 0.79) + 1 = 2
    assert R.sample(lg, 1.0, 0, 0.79, 0.62) == 0                # kept renormalised: 0.625, 0.375
    assert R.sample(lg, 1.0, 0, 0.79, 0.63) == 2
    assert R.sample_detail(lg, 1.0, 0, 0.81, 0.0)["cutoff"] == 3
    assert R.sample_detail(lg, 1.0, 0, 0.49, 0.0)["cutoff"] == 1
    assert R.sample_detail(lg, 1.0, 2, 0.99, 0.0)["cutoff"] == 2   # top-k caps the cutoff
    # temperature 0.5 on logits [2, 1, 0]: p proportional to [e^4, e^2, 1]
    z = np.exp([4.0, 2.0, 0.0]); z /= z.sum()
    assert R.sample(np.array([2.0, 1.0, 0.0]), 0.5, 0, 1.0, z[0] - 1e-9) == 0
    assert R.sample(np.array([2.0, 1.0, 0.0]), 0.5, 0, 1.0, z[0] + 1e-9) == 1
    assert R.sample(np.array([2.0, 1.0, 0.0]), 0.5, 0, 1.0, z[0] + z[1] + 1e-9) == 2


def test_sample_kept_set_matches_sorted_brute_force():
    rng = np.random.default_rng(11)
    for trial in range(20):
        lg = rng.normal(size=300) * 2
        T, k, tp = [0.7, 1.0, 1.3][trial % 3], [0, 50, 5][trial % 3], [0.9, 0.5, 0.99][trial % 3]
        e = [math.exp(v / T) for v in lg]
        z = sum(e)
        pairs = sorted(((e[i] / z, i) for i in range(len(e))), key=lambda t: (-t[0], t[1]))
        acc, kept = 0.0, []
        for pr, i in pairs:
            kept.append(i)
            acc += pr
            if acc >= tp:
                break
        if k > 0:
            kept = kept[:k]
        d = R.sample_detail(lg, T, k, tp, 0.0)
        assert list(d["kept"]) == kept


def test_sample_draw_frequencies_follow_kept_probabilities():
    lg = np.random.default_rng(12).normal(size=64)
    d = R.sample_detail(lg, 0.7, 50, 0.9, 0.0)
    p = np.exp(lg / 0.7); p /= p.sum()
    kept = d["kept"]
    q = p[kept] / p[kept].sum()
    n = 200000
    counts = {}
    for i in range(n):                                   # stratified u: exact up to 1/n
        j = R.sample(lg, 0.7, 50, 0.9, (i + 0.5) / n)
        counts[j] = counts.get(j, 0) + 1
    assert set(counts) <= set(kept.tolist())
    for i, tok in enumerate(kept):
        assert abs(counts.get(int(tok), 0) / n - q[i]) <= 2.0 / n


def test_sample_full_distribution_when_nothing_is_cut():
    lg = np.random.default_rng(13).normal(size=50)
    d = R.sample_detail(lg, 1.0, 50, 1.01, 0.0)
    assert d["cutoff"] == 50


# ------------------------------------------------------------------ Philox4x32-10
def _kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                v = [int(t, 16) for t in line.split()]
                rows.append((v[:4], v[4:6], tuple(v[6:])))
    return rows


def test_philox_known_answer_vectors():
    for ctr, key, out in _kat():
        assert R.philox4x32_10(ctr, key) == out


def _curand():
    for name in ("libcurand.so", "libcurand.so.10", ctypes.util.find_library("curand")):
        if not name:
            continue
        try:
            return ctypes.CDLL(name)
        except OSError:
            pass
    for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib"):
        try:
            return ctypes.CDLL(os.path.join(d, "libcurand.so"))
        except OSError:
            pass
    return None


def test_philox_matches_curand_host_generator():
    """cuRAND's host PHILOX4_32_10 stream: key = 64-bit seed, group g of 4 words = counter (0, 0, g, 0)."""
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    for seed in (0, 1, 0x123456789ABCDEF0, 2**64 - 1):
        gen = ctypes.c_void_p()
        if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:
            pytest.skip("cuRAND host generator unavailable")
        lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed))
        buf = (ctypes.c_uint32 * 64)()
        assert lib.curandGenerate(gen, buf, ctypes.c_size_t(64)) == 0
        lib.curandDestroyGenerator(gen)
        mine = []
        for g in range(16):
            mine += R.philox4x32_10((0, 0, g, 0), (seed & R.M32, seed >> 32))
        assert list(buf) == mine


def test_sampling_uniform_is_a_24_bit_fraction():
    for seed in (0, 5, 63):
        for step in (0, 1, 2**32 + 3):
            u = R.sampling_uniform(seed, step)
            assert 0.0 <= u < 1.0 and (u * 2**24) == int(u * 2**24)
            assert float(np.float32(u)) == u


# ------------------------------------------------------------------ generator sanity
def test_synth_is_deterministic_and_scaled():
    a = synth.normal_bf16(0, 5, 100000, 0.02)
    b = synth.normal_bf16(0, 5, 100000, 0.02)
    assert a.view(np.int16 if False else a.dtype).equal(b)
    f = synth.bf16_to_f32(a).numpy()
    assert abs(f.std() - 0.02) < 5e-4 and abs(f.mean()) < 5e-4
    c = synth.normal_bf16(0, 5, 1000, 0.02, start=50000)
    assert c.equal(a[50000:51000])
    ids = synth.token_ids(0, 0, 10000, 151936)
    assert int(ids.min()) >= 0 and int(ids.max()) < 151936


# ---------------------------------------------------------------- weight-only int8 (reading of the
# article's "What the script leaves out" section: per-output-channel symmetric int8)
def test_int8_quantiser_worked_example_with_half_even_ties():
    # max |w| = 127/128 makes the scale exactly 2^-7, so w / scale is exact and the ties are real
    row = np.array([[127 / 128, 0.5, 64.5 / 128, 65.5 / 128, -1.5 / 128, -0.5 / 128, 0.0, -127 / 128]])
    q, s = R.quantize_rows_int8(row)
    assert s.dtype == np.float32 and s[0] == np.float32(2.0 ** -7)
    assert q.tolist() == [[127, 64, 64, 66, -2, 0, 0, -127]]
    # max |w| = 1.0: t = 1/127 rounds up to the power of two 2^-6, codes on that step
    q, s = R.quantize_rows_int8(np.array([[1.0, -0.5, 0.25, 3 / 128]]))
    assert s[0] == np.float32(2.0 ** -6) and q.tolist() == [[64, -32, 16, 2]]


def test_int8_power_of_two_scale_rule():
    t = np.array([2.0 ** -7, 1.0001 * 2.0 ** -7, 0.9999 * 2.0 ** -7, 3.0, 0.0], np.float32)
    assert R.pow2_ceil(t).tolist() == [2.0 ** -7, 2.0 ** -6, 2.0 ** -7, 4.0, 0.0]


def test_int8_quantiser_bounds_and_zero_rows():
    rng = np.random.default_rng(5)
    w = rng.normal(0, 0.02, size=(64, 96)).astype(np.float32)
    w[3] = 0.0
    q, s = R.quantize_rows_int8(w)
    assert q.dtype == np.int8 and np.abs(q.astype(np.int32)).max() <= 127
    assert s[3] == 0 and not q[3].any()
    nz = s > 0
    # scales are powers of two with max/127 <= scale < 2 max/127, so the row's largest code is in [64, 127]
    m, _ = np.frexp(s[nz])
    assert (m == 0.5).all()
    amax = np.abs(w[nz]).max(axis=1)
    assert ((amax / 127 <= s[nz] * (1 + 1e-6)) & (s[nz] < 2 * amax / 127)).all()
    top = np.abs(q[nz].astype(np.int32)).max(axis=1)
    assert ((top >= 64) & (top <= 127)).all()
    # rounding to the nearest code: |w - q s| <= s / 2, exactly (the division is by a power of two)
    deq = R.dequantize_rows_int8(q, s)
    assert (np.abs(w.astype(np.float64) - deq) <= s.astype(np.float64)[:, None] / 2).all()
    # the dequantised weights are exactly representable in bf16
    assert np.array_equal(R.round_to_bf16(deq), deq)
    # a power-of-two rescale of the input rescales the scale and keeps the codes
    q2, s2 = R.quantize_rows_int8(w * np.float32(4.0))
    assert (q2 == q).all() and np.array_equal(s2, 4 * s)


def test_int8_oracle_replaces_projections_and_embedding_only(tiny_shape):
    w = synth.make_weights(tiny_shape, seed=3)
    o16 = R.Qwen3Oracle(w, tiny_shape)
    o8 = R.Qwen3Oracle(w, tiny_shape, weight_bits=8)
    for name, v in o16.W.items():
        if name == "model.embed_tokens.weight" or name.endswith(R.QUANTISED_SUFFIXES):
            q, s = R.quantize_rows_int8(w[name])
            assert np.array_equal(o8.W[name], R.dequantize_rows_int8(q, s)), name
            assert not np.array_equal(o8.W[name], v), name
        else:
            assert np.array_equal(o8.W[name], v), name
