"""The C-ABI library builds, loads and exports every symbol include/qwdecode.h
declares; argument checks that need no GPU reject bad input.  CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qwdecode.h")


@pytest.fixture(scope="module")
def lib():
    from transformer_decode_qwen3_gb300 import build, binding
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qw_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for must in ("qw_init", "qw_destroy", "qw_kv_create", "qw_kv_destroy", "qw_prefill", "qw_decode_step",
                 "qw_sample", "qw_check", "qw_last_error_message"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared in qwdecode.h but not exported"


def test_binding_covers_every_declared_symbol():
    from transformer_decode_qwen3_gb300 import binding
    assert set(declared_functions()) <= set(binding.EXPORTED)


def test_config_default_is_qwen3_0_6b(lib):
    from transformer_decode_qwen3_gb300 import binding
    cfg = binding.QwConfig()
    lib.qw_config_default(ctypes.byref(cfg))
    assert (cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.intermediate, cfg.vocab) == \
        (28, 1024, 16, 8, 128, 3072, 151936)
    assert abs(cfg.rms_eps - 1e-6) < 1e-12 and cfg.rope_theta == 1e6
    assert cfg.weight_bits == 16


@pytest.mark.parametrize("field,value", [("head_dim", 64), ("hidden", 1000), ("n_kv_heads", 3),
                                         ("intermediate", 100), ("vocab", 151937), ("max_batch", 0),
                                         ("max_tokens", 0), ("n_layers", 0), ("weight_bits", 4)])
def test_init_rejects_bad_config_without_touching_the_gpu(lib, field, value):
    from transformer_decode_qwen3_gb300 import binding
    cfg = binding.QwConfig()
    lib.qw_config_default(ctypes.byref(cfg))
    setattr(cfg, field, value)
    w = binding.QwWeights()
    h = ctypes.c_void_p()
    rc = lib.qw_init(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
    assert rc == binding.QW_EINVAL
    assert lib.qw_last_error_message()


@pytest.mark.parametrize("shape", [dict(hidden=2560, n_heads=32, n_kv_heads=8, intermediate=9728),    # 4B
                                   dict(hidden=4096, n_heads=32, n_kv_heads=8, intermediate=12288),   # 8B
                                   dict(n_heads=16, n_kv_heads=16),                                   # MHA
                                   dict(n_heads=16, n_kv_heads=1)])                                   # MQA
def test_init_takes_other_group_sizes(lib, shape):
    """Qwen3 sizes with four query heads per KV head, MHA and MQA pass the configuration check
    (qw_init then stops at the null weights, before any device work)."""
    from transformer_decode_qwen3_gb300 import binding
    cfg = binding.QwConfig()
    lib.qw_config_default(ctypes.byref(cfg))
    for k, v in shape.items():
        setattr(cfg, k, v)
    h = ctypes.c_void_p()
    assert lib.qw_init(ctypes.byref(cfg), ctypes.byref(binding.QwWeights()), ctypes.byref(h)) == binding.QW_EINVAL
    assert b"null weight pointer" in lib.qw_last_error_message()


@pytest.mark.parametrize("heads", [(24, 8), (32, 1), (12, 8)])
def test_init_names_an_unsupported_group_size(lib, heads):
    """Group sizes other than 1, 2, 4, 8, 16 (or n_heads not a multiple of n_kv_heads) are refused."""
    from transformer_decode_qwen3_gb300 import binding
    cfg = binding.QwConfig()
    lib.qw_config_default(ctypes.byref(cfg))
    cfg.n_heads, cfg.n_kv_heads = heads
    h = ctypes.c_void_p()
    assert lib.qw_init(ctypes.byref(cfg), ctypes.byref(binding.QwWeights()), ctypes.byref(h)) == binding.QW_EINVAL
    assert b"query heads per KV head" in lib.qw_last_error_message()


def test_generate_rejects_bad_arguments(lib):
    from transformer_decode_qwen3_gb300 import binding
    assert lib.qw_generate(None, None, None, 1, None, 0, 1, None, ctypes.c_uint64(0), None, None) == binding.QW_EINVAL


def test_null_arguments_are_rejected(lib):
    from transformer_decode_qwen3_gb300 import binding
    assert lib.qw_init(None, None, None) == binding.QW_EINVAL
    assert lib.qw_kv_create(None, 4, None) == binding.QW_EINVAL
    assert lib.qw_prefill(None, None, None, None, 1, None, None, 1, None, None) == binding.QW_EINVAL
    assert lib.qw_decode_step(None, None, None, 1, None, None, 1, None, None) == binding.QW_EINVAL
    assert lib.qw_sample(None, None, 1, None, ctypes.c_uint64(0), None, None) == binding.QW_EINVAL
    assert lib.qw_destroy(None) == binding.QW_EINVAL
    assert lib.qw_debug_gemm(None, None, None, 1, 32, 64, 0, 128, 0, None) == binding.QW_EINVAL
    assert b"bad argument" in lib.qw_last_error_message()


def test_sample_params_layout_matches_header():
    from transformer_decode_qwen3_gb300 import binding
    assert binding.SAMPLE_PARAMS_BYTES == 24
    assert binding.QwSampleParams.seed.offset == 16
