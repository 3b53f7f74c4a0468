"""Failure detection without a device fault: a bounded wait of the fused batch-1 decode kernel
is made to run out (the test hook asks one grid-wide exchange for an arrival that never comes,
with a 2 ms limit).  The step must give up everywhere, qw_check must report QW_ETIMEOUT, and
the context must keep working: the next step reproduces the logits of the step before the
fault bit for bit (the fused kernel adds in a fixed order)."""
import pytest
import torch

from transformer_decode_qwen3_gb300 import synth

pytestmark = pytest.mark.gpu


def test_injected_timeout_is_reported_and_the_context_survives():
    from transformer_decode_qwen3_gb300 import binding as bd
    shape = synth.ModelShape(n_layers=2)            # Qwen3-0.6B layer shape: the fused kernel takes it
    model = bd.Model(synth.make_weights(shape, device="cuda"), shape, max_batch=1, max_tokens=64)
    kv = bd.KVPool(model, 4)
    bt = torch.arange(4, dtype=torch.int32, device="cuda").view(1, 4)
    T = 5
    ids = synth.token_ids(0, 0, T, shape.vocab).cuda()
    model.prefill(ids, torch.arange(T, dtype=torch.int32, device="cuda"), [0, T], kv, bt, None)
    tok = torch.tensor([11], dtype=torch.int32, device="cuda")
    pos = torch.tensor([T], dtype=torch.int32, device="cuda")
    model.set_decode_path(2)
    try:
        before = torch.empty(1, shape.vocab, device="cuda")
        model.decode_step(tok, pos, kv, bt, before)
        assert model.check_code() == bd.QW_OK
        model.inject_timeout()
        faulted = torch.empty(1, shape.vocab, device="cuda")
        model.decode_step(tok, pos, kv, bt, faulted)
        assert model.check_code() == bd.QW_ETIMEOUT
        after = torch.empty(1, shape.vocab, device="cuda")
        model.decode_step(tok, pos, kv, bt, after)
        assert model.check_code() == bd.QW_OK
        assert torch.equal(after, before)
    finally:
        model.set_decode_path(0)
    kv.close()
    model.close()
