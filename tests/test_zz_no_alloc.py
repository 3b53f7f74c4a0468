"""qw_attn_decode_noalloc: decode attention for callers that cannot allocate
device memory (a latency-critical loop where cudaMalloc/cudaFree would
synchronise the device, or a process whose memory belongs to another allocator).
It must agree with qw_attn_decode, which keeps its partials in a context
workspace, on two calls in a row (the fixed scratch array is reused, and the
first call performs the per-device set-up)."""
import numpy as np
import pytest
import torch

from transformer_decode_qwen3_gb300 import synth
from tests import qwtest as Q

pytestmark = pytest.mark.gpu
S = Q.SMALL


def test_noalloc_attention_matches_the_workspace_version():
    from transformer_decode_qwen3_gb300 import binding as bd
    model = bd.Model(synth.make_weights(S), S, max_batch=16, max_tokens=64)
    cases = [([5, 300, 2047], 1, 7), ([0, 17, 900, 4000, 31, 64, 129, 1500], 0, 8)]
    for lens, layer, seed in cases:                      # two calls in a row
        B = len(lens)
        per = -(-(max(lens) + 1) // Q.PAGE)
        n_pages = B * per + 2
        kv = bd.KVPool(model, n_pages)
        pool = kv.view()
        bt_np, pages = Q.block_tables(lens, per * Q.PAGE, n_pages, seed=seed)
        for s, L in enumerate(lens):
            k, v = Q.synth_kv(s + seed, layer, L + 1, S.n_kv_heads, device="cuda")
            Q.inject(pool, layer, pages[s], k, v)
        bt = torch.from_numpy(bt_np).cuda()
        g = torch.Generator().manual_seed(seed)
        q = torch.randn(B, S.n_heads, 128, generator=g).cuda()
        pos = torch.tensor(lens, dtype=torch.int32, device="cuda")
        ref = torch.empty(B, S.n_heads * 128, dtype=torch.bfloat16, device="cuda")
        model.attn_decode(q, pos, kv, layer, bt, ref)
        got = torch.full_like(ref, float("nan"))
        bd.attn_decode_noalloc(q, pos, S.n_heads, S.n_kv_heads, kv.base + layer * kv.layer_stride, kv.n_pages, bt,
                               got)
        torch.cuda.synchronize()
        model.check()
        err = Q.rel_l2_rows(got.float().cpu().numpy(), ref.float().cpu().numpy())
        assert np.isfinite(err).all() and err.max() < Q.HIDDEN_TOL, f"lens {lens}: rel L2 {err.max():.2e}"
        kv.close()
    # a request beyond the fixed scratch is refused before anything is launched
    big = torch.zeros(8066 // S.n_heads + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(bd.QwError) as e:
        bd.attn_decode_noalloc(torch.zeros(big.numel(), S.n_heads, 128, device="cuda"), big, S.n_heads,
                               S.n_kv_heads, kv.base, kv.n_pages, torch.zeros(big.numel(), 1, dtype=torch.int32,
                                                                               device="cuda"),
                               torch.empty(big.numel(), S.n_heads * 128, dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == bd.QW_EINVAL
    model.close()
