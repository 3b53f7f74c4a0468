"""End-to-end parity of the CUDA path against the CPU oracle on a small model
(2 layers, hidden 256, 4 query / 2 KV heads of 128), plus the sampler on
seeded logits and the device-side error reporting."""
import numpy as np
import pytest
import torch

from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth
from tests import qwtest as Q

pytestmark = pytest.mark.gpu
S = Q.SMALL
CANARY = 1024.0     # exactly representable in bf16; marks pool slots nothing may write


@pytest.fixture(scope="module")
def small():
    from transformer_decode_qwen3_gb300 import binding
    w = synth.make_weights(S, seed=0)
    model = binding.Model(w, S, max_batch=8, max_tokens=512, debug_hidden=True)
    return binding, w, model, R.Qwen3Oracle(w, S)


def _prefill_inputs(lens, call=0, start=None):
    start = start or [0] * len(lens)
    ids = synth.token_ids(0, call, sum(lens), S.vocab)
    pos = torch.cat([torch.arange(s0, s0 + L, dtype=torch.int32) for s0, L in zip(start, lens)])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return ids, pos, cu


def _hidden(model, n):
    out = []
    for layer in range(S.n_layers):
        buf = torch.empty(n, S.hidden, device="cuda")
        model.debug_hidden(layer, buf, n)
        out.append(buf.cpu().double().numpy())
    return out


def test_prefill_ragged_then_decode(small):
    bd, w, model, orc = small
    lens, cap, steps = [1, 70, 130], 160, 4
    n_pages = 3 * (cap // Q.PAGE) + 7
    kv = bd.KVPool(model, n_pages)
    pool = kv.view()
    pool.fill_(CANARY)
    bt_np, pages = Q.block_tables(lens, cap, n_pages, seed=1)
    bt = torch.from_numpy(bt_np).cuda()
    ids, pos, cu = _prefill_inputs(lens)
    last = torch.empty(len(lens), S.vocab, device="cuda")
    model.prefill(ids.cuda(), pos.cuda(), cu, kv, bt, last)
    model.check()
    hid = _hidden(model, int(cu[-1]))
    caches = []
    for s, L in enumerate(lens):
        cache, h_ref = orc.new_cache(), []
        ref = orc.forward(ids[cu[s]:cu[s + 1]].numpy(), np.arange(L), cache, hiddens=h_ref)
        caches.append(cache)
        for layer in range(S.n_layers):
            err = Q.rel_l2_rows(hid[layer][cu[s]:cu[s + 1]], h_ref[layer])
            assert err.max() < Q.HIDDEN_TOL, f"seq {s} layer {layer}: hidden rel L2 {err.max():.2e}"
        err = Q.rel_l2_rows(last[s:s + 1].cpu().numpy(), ref[-1:])
        assert err.max() < Q.LOGIT_TOL, f"seq {s}: last logits rel L2 {err.max():.2e}"
        # the cache holds the rotated keys and the values at exactly their positions
        for layer in range(S.n_layers):
            k, v = Q.read_kv(pool, layer, pages[s], L)
            kr, vr = cache[layer].k.transpose(1, 0, 2), cache[layer].v.transpose(1, 0, 2)
            assert Q.rel_l2_rows(k.reshape(L, -1), kr.reshape(L, -1)).max() < Q.HIDDEN_TOL
            assert Q.rel_l2_rows(v.reshape(L, -1), vr.reshape(L, -1)).max() < Q.HIDDEN_TOL
    # untouched slots keep the canary: bookkeeping is exact
    used = torch.zeros(n_pages, Q.PAGE, dtype=torch.bool)
    for s, L in enumerate(lens):
        for p in range(L):
            used[pages[s][p // Q.PAGE], p % Q.PAGE] = True
    slots = pool.permute(1, 4, 0, 2, 3, 5)                # [page, slot, layer, K/V, n_kv, 128]
    assert bool((slots[~used.cuda()].float() == CANARY).all())
    assert not bool((slots[used.cuda()].float() == CANARY).any())

    # decode steps, teacher-forced with fixed tokens; batch = the three sequences
    logits = torch.empty(len(lens), S.vocab, device="cuda")
    toks_all = synth.token_ids(0, 1, steps * len(lens), S.vocab).view(steps, len(lens))
    for step in range(steps):
        toks = toks_all[step]
        p = torch.tensor([L + step for L in lens], dtype=torch.int32)
        model.decode_step(toks.cuda(), p.cuda(), kv, bt, logits)
        model.check()
        hid = _hidden(model, len(lens))
        for s in range(len(lens)):
            h_ref = []
            ref = orc.forward([int(toks[s])], [int(p[s])], caches[s], hiddens=h_ref)
            err = Q.rel_l2_rows(logits[s:s + 1].cpu().numpy(), ref)
            assert err.max() < Q.LOGIT_TOL, f"step {step} seq {s}: logits rel L2 {err.max():.2e}"
            for layer in range(S.n_layers):
                assert Q.rel_l2_rows(hid[layer][s:s + 1], h_ref[layer]).max() < Q.HIDDEN_TOL


def test_chunked_prefill_equals_one_prefill(small):
    bd, w, model, orc = small
    L1, L2 = 40, 30
    kv = bd.KVPool(model, 16)
    bt_np, pages = Q.block_tables([0], 80, 16, seed=2)
    bt = torch.from_numpy(bt_np).cuda()
    ids, _, _ = _prefill_inputs([L1 + L2], call=5)
    a = torch.empty(1, S.vocab, device="cuda")
    model.prefill(ids[:L1].cuda(), torch.arange(L1, dtype=torch.int32).cuda(), [0, L1], kv, bt, a)
    b = torch.empty(1, S.vocab, device="cuda")
    model.prefill(ids[L1:].cuda(), torch.arange(L1, L1 + L2, dtype=torch.int32).cuda(), [0, L2], kv, bt, b)
    model.check()
    ref = orc.forward(ids.numpy(), np.arange(L1 + L2), orc.new_cache())
    assert Q.rel_l2_rows(a.cpu().numpy(), ref[L1 - 1:L1]).max() < Q.LOGIT_TOL
    assert Q.rel_l2_rows(b.cpu().numpy(), ref[-1:]).max() < Q.LOGIT_TOL


def test_sampler_matches_oracle_on_seeded_logits(small):
    bd, w, model, orc = small
    B, V = 8, S.vocab
    g = torch.Generator().manual_seed(11)
    logits = torch.randn(B, V, generator=g) * 2.0
    logits[3, 17] = logits[3, 901] = 50.0                  # an exact tie: lowest id must win
    rows = [(0.0, 1, 1.0, 0), (0.7, 50, 0.9, 1), (1.0, 1, 0.5, 2), (0.0, 50, 0.9, 3), (1.3, 1024, 0.95, 4),
            (0.5, 5, 1.0, 5), (0.9, 200, 0.3, 6), (2.0, 1000, 1.0, 7)]
    params = bd.sample_params(rows)
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    for counter in (0, 1, 12345, 2**33 + 5):
        model.sample(params, counter, out, logits=logits.cuda())
        model.check()
        got = out.cpu().numpy()
        for r, (t, k, p, seed) in enumerate(rows):
            u = R.sampling_uniform(seed, counter)
            d = R.sample_detail(logits[r].numpy(), t, k, p, u)
            if t == 0.0:
                assert got[r] == d["id"]
            elif not Q.sample_exempt(d, p):
                assert got[r] == d["id"], f"row {r} counter {counter}: gpu {got[r]} vs oracle {d['id']}"
    assert out.cpu().numpy()[3] == 17


def test_device_errors_are_reported_and_the_context_survives(small):
    bd, w, model, orc = small
    kv = bd.KVPool(model, 8)
    bt = torch.arange(8, dtype=torch.int32).view(1, 8).cuda()
    logits = torch.empty(1, S.vocab, device="cuda")
    one = lambda v: torch.tensor([v], dtype=torch.int32, device="cuda")
    model.decode_step(one(S.vocab), one(0), kv, bt, logits)          # token id out of range
    assert model.check_code() == bd.QW_ERANGE
    model.decode_step(one(3), one(8 * Q.PAGE), kv, bt, logits)       # position past the block table
    assert model.check_code() == bd.QW_ERANGE
    bad = bt.clone()
    bad[0, 0] = 1000                                                  # page id outside the pool
    model.decode_step(one(3), one(0), kv, bad, logits)
    assert model.check_code() == bd.QW_ERANGE
    model.decode_step(one(3), one(0), kv, bt, logits)                 # a valid call still works
    assert model.check_code() == bd.QW_OK
    with pytest.raises(bd.QwError):                                   # empty sequence: rejected on the host
        model.prefill(one(3), one(0), [0, 0], kv, bt, logits)


@pytest.mark.parametrize("variant", [0, 1])
def test_prefill_attention_kernels_match_oracle(small, variant):
    """The tcgen05 flash kernel (0) and the mma.sync one (1), ragged lengths across tile edges."""
    bd, w, model, orc = small
    lens = [1, 63, 65, 127, 129, 100]         # 485 tokens <= max_tokens; 1 and 2 key tiles, ragged q tiles
    cap = 144
    n_pages = len(lens) * (cap // Q.PAGE)
    kv = bd.KVPool(model, n_pages)
    bt_np, _ = Q.block_tables(lens, cap, n_pages, seed=3)
    ids, pos, cu = _prefill_inputs(lens, call=9)
    last = torch.empty(len(lens), S.vocab, device="cuda")
    model.set_prefill_attention(variant)
    try:
        model.prefill(ids.cuda(), pos.cuda(), cu, kv, torch.from_numpy(bt_np).cuda(), last)
        model.check()
    finally:
        model.set_prefill_attention(0)
    for s, L in enumerate(lens):
        ref = orc.forward(ids[cu[s]:cu[s + 1]].numpy(), np.arange(L), orc.new_cache(), last_only=True)
        err = Q.rel_l2_rows(last[s:s + 1].cpu().numpy(), ref)
        assert err.max() < Q.LOGIT_TOL, f"variant {variant} seq {s} (L={L}): {err.max():.2e}"


def test_mixed_prefill_and_decode_in_one_call(small):
    """One qw_prefill call carries a fresh prompt, a prompt chunk appended to a cached prefix,
    and two decode tokens (one-token chunks at the position after their caches), each sequence
    reading only its own pages; every sequence's last logits equal the oracle's over its whole
    history, and the decode rows equal what qw_decode_step gives for the same tokens."""
    bd, w, model, orc = small
    # sequences: 0 fresh prompt of 37; 1 has 50 cached, adds a chunk of 20; 2 and 3 have 64 and
    # 9 cached and decode one token each
    hist = [0, 50, 64, 9]
    new = [37, 20, 1, 1]
    cap = 96
    n_pages = 4 * (cap // Q.PAGE) + 3
    kv = bd.KVPool(model, n_pages)
    bt_np, _ = Q.block_tables(hist, cap, n_pages, seed=12)
    bt = torch.from_numpy(bt_np).cuda()
    ids_all = [synth.token_ids(0, 40 + s, hist[s] + new[s], S.vocab) for s in range(4)]
    # the cached prefixes, written by one prefill of sequences 1..3
    pre = [s for s in range(4) if hist[s]]
    ids = torch.cat([ids_all[s][:hist[s]] for s in pre])
    pos = torch.cat([torch.arange(hist[s], dtype=torch.int32) for s in pre])
    cu = np.concatenate([[0], np.cumsum([hist[s] for s in pre])]).astype(np.int32)
    model.prefill(ids.cuda(), pos.cuda(), cu, kv, bt[pre].contiguous(), torch.empty(len(pre), S.vocab, device="cuda"))
    model.check()
    # the mixed call
    ids = torch.cat([ids_all[s][hist[s]:] for s in range(4)])
    pos = torch.cat([torch.arange(hist[s], hist[s] + new[s], dtype=torch.int32) for s in range(4)])
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    last = torch.empty(4, S.vocab, device="cuda")
    model.prefill(ids.cuda(), pos.cuda(), cu, kv, bt, last)
    model.check()
    for s in range(4):
        L = hist[s] + new[s]
        ref = orc.forward(ids_all[s].numpy(), np.arange(L), orc.new_cache(), last_only=True)
        err = Q.rel_l2_rows(last[s:s + 1].cpu().numpy(), ref).max()
        assert err < Q.LOGIT_TOL, f"sequence {s}: logits rel L2 {err:.2e}"
    # the decode rows as a decode step (same positions: the step rewrites the same cache slots)
    rows = [2, 3]
    dec = torch.empty(2, S.vocab, device="cuda")
    model.decode_step(torch.tensor([int(ids_all[s][-1]) for s in rows], dtype=torch.int32).cuda(),
                      torch.tensor([hist[s] for s in rows], dtype=torch.int32).cuda(), kv, bt[rows].contiguous(), dec)
    model.check()
    assert Q.rel_l2_rows(dec.cpu().numpy(), last[rows].cpu().numpy()).max() < Q.LOGIT_TOL
    kv.close()
