"""Pins of the plain single-precision C oracle (oracle/qwen3_ref.c).  CPU only.

Two kinds of pin: direct ones against closed forms, worked examples and the published
Philox vectors (the same facts the numpy oracle is pinned to), and agreement with the
float64 numpy oracle, itself pinned, on whole forward passes (tiny shape, and two layers of
the full Qwen3-0.6B widths) to float32 rounding."""
import math
import os

import numpy as np
import pytest

from oracle import qwen3_c as C
from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lib():
    return C.load()


def _bf16(vals):
    import torch
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


# ------------------------------------------------------------------ direct pins
def test_rmsnorm_worked_values(lib):
    np.testing.assert_allclose(C.rms_norm([3.0, 4.0], _bf16([1.0, 1.0])), [0.8485281374, 1.1313708499], rtol=1e-6)
    np.testing.assert_allclose(C.rms_norm(np.full(8, 1e-3), _bf16([1.0] * 8)), 1 / math.sqrt(2), rtol=1e-6)
    np.testing.assert_allclose(C.rms_norm([3.0, 4.0], _bf16([2.0, -0.5])), [1.6970562748, -0.5656854249],
                               rtol=1e-6)


def test_rope_identity_norms_and_half_split_basis(lib):
    x = np.random.default_rng(1).normal(size=128).astype(np.float32)
    np.testing.assert_array_equal(C.rope(x, 0), x)
    for pos in (1, 7, 32799):
        y = C.rope(x, pos)
        np.testing.assert_allclose(np.hypot(y[:64], y[64:]), np.hypot(x[:64], x[64:]), rtol=1e-6)
    for i in (0, 5, 63):
        f = 10.0 ** (-6 * i / 64)
        e = np.zeros(128, dtype=np.float32)
        e[i] = 1.0
        y = C.rope(e, 3)
        np.testing.assert_allclose([y[i], y[i + 64]], [math.cos(3 * f), math.sin(3 * f)], atol=1e-6)
        e = np.zeros(128, dtype=np.float32)
        e[i + 64] = 1.0
        y = C.rope(e, 3)
        np.testing.assert_allclose([y[i], y[i + 64]], [-math.sin(3 * f), math.cos(3 * f)], atol=1e-6)


def test_philox_known_answer_vectors(lib):
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        rows = [[int(t, 16) for t in line.split()] for line in f if line.strip() and not line.startswith("#")]
    assert rows
    for v in rows:
        assert C.philox4x32_10(v[:4], v[4:6]) == tuple(v[6:])
    u = C.sampling_uniform(7, 3)
    assert 0.0 <= u < 1.0 and (u * 2 ** 24).is_integer()


def test_sample_worked_example_and_greedy(lib):
    lg = np.log([0.5, 0.2, 0.3])
    d = C.sample_detail(lg, 1.0, 0, 0.79, 0.0)
    assert d["cutoff"] == 2 and d["id"] == 0
    assert C.sample_detail(lg, 1.0, 0, 0.79, 0.62)["id"] == 0       # kept renormalised: 0.625, 0.375
    assert C.sample_detail(lg, 1.0, 0, 0.79, 0.63)["id"] == 2
    assert C.sample_detail(lg, 1.0, 0, 0.81, 0.0)["cutoff"] == 3
    assert C.sample_detail(lg, 1.0, 2, 0.99, 0.0)["cutoff"] == 2     # top-k caps the cutoff
    tie = np.zeros(10)
    tie[[3, 6]] = 1.0
    assert C.sample_detail(tie, 0.0, 0, 1.0, 0.0)["id"] == 3          # lowest id wins a tie


def test_sample_kept_mass_matches_sorted_brute_force(lib):
    rng = np.random.default_rng(11)
    for trial in range(12):
        lg = (rng.normal(size=300) * 2).astype(np.float32)
        T, k, tp = [0.7, 1.0, 1.3][trial % 3], [0, 50, 5][trial % 3], [0.9, 0.5, 0.99][trial % 3]
        e = np.exp(lg.astype(np.float64) / T)
        p = e / e.sum()
        order = sorted(range(len(p)), key=lambda i: (-p[i], i))
        acc, kept = 0.0, []
        for i in order:
            kept.append(i)
            acc += p[i]
            if acc >= tp:
                break
        if k > 0:
            kept = kept[:k]
        for u in (0.0, 0.37, 0.999):
            d = C.sample_detail(lg, T, k, tp, u)
            assert d["cutoff"] == len(kept)
            np.testing.assert_allclose(d["cum_at_cutoff"], p[kept].sum(), rtol=1e-6)
            q = np.cumsum(p[kept]) / p[kept].sum()
            assert d["id"] == kept[int(np.searchsorted(q, u, side="right"))]


# ------------------------------------------------------------------ whole passes
def _pair(shape, seed=0):
    w = synth.make_weights(shape, seed=seed)
    return C.COracle(w, shape), R.Qwen3Oracle(w, shape)


def test_forward_with_cache_agrees_with_numpy_oracle(tiny_shape):
    c, r = _pair(tiny_shape)
    cc, rc = c.new_cache(16), r.new_cache()
    ids = [11, 200, 3, 3, 42, 255, 0, 17]
    for sl in (slice(0, 5), slice(5, 6), slice(6, 8)):          # prefill, decode, chunk
        pos = np.arange(sl.start, sl.stop)
        got, hid = c.forward(ids[sl], pos, cc, hiddens=True)
        h_ref = []
        ref = r.forward(ids[sl], pos, rc, hiddens=h_ref)
        assert _rel(got, ref) < 2e-6
        for layer in range(tiny_shape.n_layers):
            assert _rel(hid[layer], h_ref[layer]) < 2e-6
    assert cc.len == 8


def test_cached_decode_equals_full_recompute(tiny_shape):
    c, _ = _pair(tiny_shape)
    ids = [11, 200, 3, 3, 42, 255, 0, 17]
    full = c.forward(ids, np.arange(8), c.new_cache(8))
    cache = c.new_cache(8)
    rows = [c.forward(ids[:5], np.arange(5), cache)[-1]]
    for t in range(5, 8):
        rows.append(c.forward([ids[t]], [t], cache)[-1])
    np.testing.assert_allclose(np.array(rows), full[4:], rtol=2e-5, atol=1e-6)


def test_two_full_width_layers_agree_with_numpy_oracle():
    shape = synth.ModelShape(n_layers=2)
    c, r = _pair(shape)
    ids = synth.token_ids(0, 5, 6, shape.vocab).numpy()
    cc, rc = c.new_cache(8), r.new_cache()
    got = c.forward(ids, np.arange(6), cc, last_only=True)
    ref = r.forward(ids, np.arange(6), rc, last_only=True)
    assert _rel(got, ref) < 1e-5
    got = c.forward([int(ids[0])], [6], cc, last_only=True)
    ref = r.forward([int(ids[0])], [6], rc, last_only=True)
    assert _rel(got, ref) < 1e-5


def test_generate_agrees_with_numpy_oracle_and_recompute(tiny_shape):
    c, r = _pair(tiny_shape)
    prompt = [3, 77, 200, 5]
    for temp, k, tp in ((0.0, 0, 1.0), (1.3, 0, 0.9), (0.8, 5, 1.0)):
        ids, rows = c.generate(prompt, 5, temp, k, tp, seed=9)
        ids_r, rows_r = R.generate(r, prompt, 5, temperature=temp, top_k=k, top_p=tp, seed=9)
        assert ids == ids_r
        assert _rel(rows, np.array(rows_r)) < 2e-6
        # decode position T + i - 1: each row equals the last row of a full recompute
        ref = c.forward(prompt + ids[:4], np.arange(8), c.new_cache(8))[-1]
        np.testing.assert_allclose(rows[4], ref, rtol=2e-5, atol=1e-6)


def test_int8_weights_agree_with_numpy_oracle(tiny_shape):
    """The C oracle run on the int8-dequantised weights (exact bf16 values, as the benchmark's
    CPU baseline builds them) agrees with the numpy oracle's own weight_bits = 8 mode."""
    import torch
    w = synth.make_weights(tiny_shape, seed=4)
    w8 = dict(w)
    for name in w:
        if name == "model.embed_tokens.weight" or name.endswith(R.QUANTISED_SUFFIXES):
            deq = R.dequantize_rows_int8(*R.quantize_rows_int8(w[name]))
            assert np.array_equal(R.round_to_bf16(deq), deq)            # exact in bf16
            w8[name] = torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16)
    c = C.COracle(w8, tiny_shape)
    r = R.Qwen3Oracle(w, tiny_shape, weight_bits=8)
    ids = [11, 200, 3, 3, 42, 255, 0, 17]
    got = c.forward(ids, np.arange(8), c.new_cache(8))
    ref = r.forward(ids, np.arange(8), r.new_cache())
    assert _rel(got, ref) < 2e-6
