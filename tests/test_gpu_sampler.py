"""qw_sample against the oracle's sample() (the article, Step 8) on full-vocabulary rows
(151,936 logits), including the article's own call: top-p with no top-k cap, whatever the
size of the nucleus.  Ids must equal the oracle's except for draws the parity rules exempt
(the draw within 1e-3 of a cumulative boundary, or the cutoff within 1e-3 of top_p); an
exempt draw must still be a valid inverse-CDF draw of u up to 2e-4 (a 100,000-entry nucleus
has boundaries ~1e-5 apart, so the exemption covers most of its draws)."""
import numpy as np
import pytest
import torch

from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth
from tests import qwtest as Q

pytestmark = pytest.mark.gpu
V = synth.QWEN3_0_6B.vocab
# one small layer in front of the full vocabulary: the sampler only sees the vocabulary size
SHAPE = synth.ModelShape(n_layers=1, hidden=256, n_heads=4, n_kv_heads=2, head_dim=128, intermediate=384, vocab=V)


@pytest.fixture(scope="module")
def model():
    from transformer_decode_qwen3_gb300 import binding as bd
    m = bd.Model(synth.make_weights(SHAPE, device="cuda"), SHAPE, max_batch=64, max_tokens=64)
    yield bd, m
    m.close()


def _check_rows(bd, m, logits, rows, counter, min_strict):
    params = bd.sample_params(rows)
    out = torch.empty(len(rows), dtype=torch.int32, device="cuda")
    m.sample(params, counter, out, logits=logits.cuda())
    m.check()
    got = out.cpu().numpy()
    strict = 0
    for r, (t, k, p, seed) in enumerate(rows):
        u = R.sampling_uniform(seed, counter)
        d = R.sample_detail(logits[r].double().numpy(), t, k, p, u)
        if t == 0.0 or not Q.sample_exempt(d, p):
            assert got[r] == d["id"], f"row {r} {rows[r]} counter {counter}: gpu {got[r]} vs oracle {d['id']}"
            strict += 1
        else:
            assert Q.sample_draw_is_valid(logits[r].numpy(), t, k, p, u, int(got[r])), \
                f"row {r} {rows[r]} counter {counter}: gpu {got[r]} is not a draw of u = {u} (oracle {d['id']})"
    assert strict >= min_strict
    return got


@pytest.mark.parametrize("std", [0.5, 2.0])
def test_uncapped_top_p_and_caps_match_oracle(model, std):
    """Flat (std 0.5: the nucleus holds most of the vocabulary) and peaked (std 2) rows."""
    bd, m = model
    B = 24
    g = torch.Generator().manual_seed(int(std * 10))
    logits = torch.randn(B, V, generator=g) * std
    cases = [(0.7, 0, 0.95), (1.0, 0, 0.9), (0.7, 50, 0.9), (1.0, 0, 1.0), (0.5, 1, 0.9), (1.3, 5000, 0.99),
             (0.7, 0, 0.5), (0.0, 0, 1.0)]
    rows = [(*cases[r % len(cases)], 1000 + r) for r in range(B)]
    for counter in (0, 7, 2**33 + 1):
        _check_rows(bd, m, logits, rows, counter, min_strict=B // 4)


def test_ties_resolve_to_the_lowest_ids(model):
    bd, m = model
    logits = torch.full((3, V), -20.0)
    logits[0] = 0.0                                          # every entry equal: uniform over all ids
    tied = [7, 3, 100, 151935, 42, 9000, 5, 77777, 1, 60000]
    logits[1, tied] = 5.0                                    # ten entries of 0.1 each (the rest ~1e-11)
    logits[2, [11, 12]] = 3.0                                # greedy tie
    rows = [(1.0, 0, 1.0, 1), (1.0, 0, 0.35, 2), (0.0, 0, 1.0, 3)]
    for counter in range(6):
        got = _check_rows(bd, m, logits, rows, counter, min_strict=2)
        assert got[1] in sorted(tied)[:4]                    # cutoff 4: the four lowest tied ids
        assert got[2] == 11


def test_context_logits_use_the_lm_head_tile_maxima(model):
    """Greedy and sampled rows from the context's own logits (qw_sample with logits NULL:
    the LM head's per-tile maxima) agree with the same rows passed explicitly."""
    bd, m = model
    B = 4
    kv = bd.KVPool(m, 2 * B)
    bt = torch.arange(2 * B, dtype=torch.int32, device="cuda").view(B, 2)   # each sequence its own pages
    toks = synth.token_ids(0, 11, B, V).cuda()
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    logits = torch.empty(B, V, device="cuda")
    m.set_decode_path(1)
    try:
        m.decode_step(toks, pos, kv, bt, logits)     # explicit rows
        m.decode_step(toks, pos, kv, bt, None)       # the same step, rows kept in the context
    finally:
        m.set_decode_path(0)
    rows = [(0.0, 0, 1.0, 0), (0.7, 0, 0.95, 1), (0.0, 0, 1.0, 2), (1.0, 50, 0.9, 3)]
    params = bd.sample_params(rows)
    a = torch.empty(B, dtype=torch.int32, device="cuda")
    b = torch.empty(B, dtype=torch.int32, device="cuda")
    m.sample(params, 5, a, logits=logits)
    m.sample(params, 5, b)
    m.check()
    lg = logits.cpu().numpy()
    for r, (t, k, p, seed) in enumerate(rows):
        # the two steps add their split-K partial products in different orders, so their logits
        # differ in the last bits: greedy rows agree away from near-ties, sampled rows from the
        # context must be valid draws of the explicit rows' distribution
        if t == 0.0:
            top2 = np.sort(lg[r])[-2:]
            if top2[1] - top2[0] > 1e-3:
                assert int(b[r]) == int(a[r]) == int(np.argmax(lg[r]))
        else:
            assert Q.sample_draw_is_valid(lg[r], t, k, p, R.sampling_uniform(seed, 5), int(b[r]))
    kv.close()


def test_invalid_parameters_are_reported(model):
    bd, m = model
    logits = torch.zeros(1, V, device="cuda")
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    m.sample(bd.sample_params([(1.0, -1, 0.9, 0)]), 0, out, logits=logits)
    assert m.check_code() == bd.QW_EINVAL
    m.sample(bd.sample_params([(1.0, 0, 1.5, 0)]), 0, out, logits=logits)
    assert m.check_code() == bd.QW_EINVAL
    m.sample(bd.sample_params([(1.0, 0, 0.9, 0)]), 0, out, logits=logits)
    assert m.check_code() == bd.QW_OK and 0 <= int(out) < V


def test_topk_rows_and_their_hand_over(model):
    """Rows capped by top_k <= 1024 take the one-CTA top-k kernel; a row whose bound bucket holds
    more than its candidate buffer (3000 tied maxima) or a constant row is handed to the
    general kernel.  Every row must still match the oracle."""
    bd, m = model
    g = torch.Generator().manual_seed(99)
    logits = torch.randn(8, V, generator=g) * 2.0
    logits[5, :] = torch.randn(V, generator=g) * 0.5
    logits[5, torch.randperm(V, generator=g)[:3000]] = 6.0     # 3000 tied maxima
    logits[6, :] = 1.5                                           # constant row
    rows = [(0.7, 50, 0.9, 1), (1.0, 1024, 0.95, 2), (1.0, 7, 1.0, 3), (0.3, 1, 0.5, 4), (2.0, 300, 0.99, 5),
            (1.0, 100, 0.9, 6), (1.0, 10, 1.0, 7), (0.7, 1000, 0.999, 8)]
    for counter in (0, 3, 2**40 + 5):
        got = _check_rows(bd, m, logits, rows, counter, min_strict=4)
        assert got[6] < 10                                       # uniform over the 10 lowest ids
