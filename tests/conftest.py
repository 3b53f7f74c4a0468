import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def tiny_shape():
    from transformer_decode_qwen3_gb300.synth import ModelShape
    # hidden = n_heads * head_dim so that o_proj can be the identity in closed-form pins
    return ModelShape(n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16,
                      intermediate=96, vocab=257, weight_std=0.2)
