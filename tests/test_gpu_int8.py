"""Weight-only int8 (per output channel) at full Qwen3-0.6B size against the oracle run on the
same quantised weights (Qwen3Oracle(weight_bits=8), which quantises the weights itself).

The fused batch-1 kernel streams the int8 codes; the per-op path computes with the dequantised
bf16 weights.  Decode is teacher-forced as in the bf16 workload tests.  The ids are compared wherever the
oracle's top-1 / top-2 margin exceeds 0.05; on these quantised random weights fewer steps have
such a margin than with bf16 weights, so at least a quarter of the steps must be comparable.
"""
import pytest

from oracle import qwen3_ref as R
from transformer_decode_qwen3_gb300 import synth
from tests import qwtest as Q
from tests.test_gpu_workloads import _prompt_then_greedy

pytestmark = pytest.mark.gpu
S = Q.FULL


@pytest.fixture(scope="module")
def full_int8():
    from transformer_decode_qwen3_gb300 import binding
    w = synth.make_weights(S, seed=0)
    model = binding.Model(w, S, max_batch=8, max_tokens=1024, debug_hidden=True, weight_bits=8)
    orc = R.Qwen3Oracle(w, S, weight_bits=8)
    return binding, model, orc


def test_int8_prompt5_greedy8_fused(full_int8):
    """A five-token prompt and eight greedy steps through the fused kernel streaming int8 codes."""
    _prompt_then_greedy(full_int8, 5, 8, call=0, path=2, min_checked=0.25)


def test_int8_prompt5_greedy8_per_op(full_int8):
    """The same workload through the per-op kernels (dequantised bf16 weights, every layer checked)."""
    _prompt_then_greedy(full_int8, 5, 8, call=0, path=1, min_checked=0.25)


def test_int8_prompt512_greedy32_fused(full_int8):
    _prompt_then_greedy(full_int8, 512, 32, call=1, path=2, min_checked=0.25)
