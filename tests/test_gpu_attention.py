"""Split-KV decode attention of one layer (qw_attn_decode) against the oracle's
attention core, on synthetic paged caches from 1 to 32768 positions."""
import numpy as np
import pytest
import torch

from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth
from tests import qwtest as Q

pytestmark = pytest.mark.gpu
S = Q.SMALL           # 4 query heads, 2 KV heads


@pytest.fixture(scope="module")
def model():
    from transformer_decode_qwen3_gb300 import binding
    w = synth.make_weights(S)
    return binding, binding.Model(w, S, max_batch=16, max_tokens=64)


def _case(bd, model, lens, layer=1, seed=0):
    B = len(lens)
    cap = max(lens) + 1
    per = -(-cap // Q.PAGE)
    kv = bd.KVPool(model, B * per + 3)
    pool = kv.view()
    bt_np, pages = Q.block_tables(lens, per * Q.PAGE, B * per + 3, seed=seed)
    ks, vs = [], []
    for s, L in enumerate(lens):
        k, v = Q.synth_kv(s, layer, L + 1, S.n_kv_heads, device="cuda")
        Q.inject(pool, layer, pages[s], k, v)
        ks.append(k.cpu())
        vs.append(v.cpu())
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, S.n_heads, 128, generator=g)
    out = torch.empty(B, S.n_heads * 128, dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor(lens, dtype=torch.int32)
    model.attn_decode(q.cuda(), pos.cuda(), kv, layer, torch.from_numpy(bt_np).cuda(), out)
    model.check()
    got = out.float().cpu().numpy()
    for s, L in enumerate(lens):
        kk = R.bf16_to_f64(ks[s]).transpose(1, 0, 2)
        vv = R.bf16_to_f64(vs[s]).transpose(1, 0, 2)
        ref = R.gqa_attention(q[s].double().numpy()[:, None, :], kk, vv, np.arange(L + 1), [L])
        err = Q.rel_l2_rows(got[s:s + 1], ref.reshape(1, -1))
        assert err.max() < Q.HIDDEN_TOL, f"seq {s} (L={L}): rel L2 {err.max():.2e}"
    kv.close()


def test_decode_attention_short_and_ragged(model):
    bd, m = model
    _case(bd, m, [0, 1, 15, 16, 17, 100, 511, 1000], seed=1)


def test_decode_attention_long_context(model):
    bd, m = model
    _case(bd, m, [32767, 20000, 4095], seed=2)
