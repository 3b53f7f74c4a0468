"""Other Qwen3 dense sizes and attention layouts (the article, Step 5: "From MHA to MQA to GQA"),
head_dim 128, each with 2 layers and a reduced vocabulary so the oracle stays fast:

  1.7B  hidden 2048, 16 query / 8 KV heads (2 per group), intermediate 6144
  4B    hidden 2560, 32 / 8 (4 per group), intermediate 9728
  8B    hidden 4096, 32 / 8 (4 per group), intermediate 12288
  MHA   hidden 1024, 8 / 8 (1 per group);  G8: 16 / 2;  MQA: 16 / 1 (one KV head)

Ragged prefill (query tiles of 128 / G positions), then a batched and a batch-1 decode step,
against the oracle."""
import numpy as np
import pytest
import torch

from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth
from tests import qwtest as Q

pytestmark = pytest.mark.gpu
SHAPES = {
    "1.7B": dict(hidden=2048, n_heads=16, n_kv_heads=8, intermediate=6144),
    "4B": dict(hidden=2560, n_heads=32, n_kv_heads=8, intermediate=9728),
    "8B": dict(hidden=4096, n_heads=32, n_kv_heads=8, intermediate=12288),
    "MHA": dict(hidden=1024, n_heads=8, n_kv_heads=8, intermediate=3072),
    "G8": dict(hidden=1024, n_heads=16, n_kv_heads=2, intermediate=3072),
    "MQA": dict(hidden=1024, n_heads=16, n_kv_heads=1, intermediate=3072),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_other_sizes_and_layouts_prefill_and_decode(name):
    from transformer_decode_qwen3_gb300 import binding as bd
    S = synth.ModelShape(n_layers=2, head_dim=128, vocab=8192, **SHAPES[name])
    w = synth.make_weights(S, seed=5)
    model = bd.Model(w, S, max_batch=4, max_tokens=512)
    orc = R.Qwen3Oracle(w, S)
    lens, cap = [7, 150, 300], 320
    n_pages = 3 * (cap // Q.PAGE) + 3
    kv = bd.KVPool(model, n_pages)
    bt_np, _ = Q.block_tables(lens, cap, n_pages, seed=9)
    bt = torch.from_numpy(bt_np).cuda()
    ids = synth.token_ids(5, 0, sum(lens), S.vocab)
    pos = torch.cat([torch.arange(L, dtype=torch.int32) for L in lens])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    last = torch.empty(len(lens), S.vocab, device="cuda")
    model.prefill(ids.cuda(), pos.cuda(), cu, kv, bt, last)
    model.check()
    caches = []
    for s, L in enumerate(lens):
        cache = orc.new_cache()
        ref = orc.forward(ids[cu[s]:cu[s + 1]].numpy(), np.arange(L), cache, last_only=True)
        caches.append(cache)
        assert Q.rel_l2_rows(last[s:s + 1].cpu().numpy(), ref).max() < Q.LOGIT_TOL
    # one batched decode step (split-operand projections), then batch 1 on the last sequence
    toks = synth.token_ids(5, 1, len(lens), S.vocab)
    logits = torch.empty(len(lens), S.vocab, device="cuda")
    model.decode_step(toks.cuda(), torch.tensor(lens, dtype=torch.int32).cuda(), kv, bt, logits)
    model.check()
    for s, L in enumerate(lens):
        ref = orc.forward([int(toks[s])], [L], caches[s], last_only=True)
        assert Q.rel_l2_rows(logits[s:s + 1].cpu().numpy(), ref).max() < Q.LOGIT_TOL
    s, L = 2, lens[2] + 1
    tok = torch.tensor([3], dtype=torch.int32, device="cuda")
    one = torch.empty(1, S.vocab, device="cuda")
    model.decode_step(tok, torch.tensor([L], dtype=torch.int32, device="cuda"), kv, bt[s:s + 1], one)
    model.check()
    ref = orc.forward([3], [L], caches[s], last_only=True)
    assert Q.rel_l2_rows(one.cpu().numpy(), ref).max() < Q.LOGIT_TOL
    kv.close()
    model.close()
