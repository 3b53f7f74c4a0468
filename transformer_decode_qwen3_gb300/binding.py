"""ctypes binding of libqwdecode (include/qwdecode.h).

Argument marshalling only: every step of the forward pass and the sampler runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.  The
functions keep the C names (qw_init, qw_prefill, qw_decode_step, qw_sample, ...);
:class:`Model` and :class:`KVPool` wrap them for torch tensors.

Loading fails loudly when the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .synth import ModelShape, weight_names

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libqwdecode.so")

QW_OK, QW_EINVAL, QW_ERANGE, QW_ENOMEM, QW_EKVFULL, QW_ECUDA, QW_ETIMEOUT = 0, -1, -2, -3, -4, -5, -6
QW_PAGE_SIZE = 16
QW_HEAD_DIM = 128
QW_TRACE_SLOTS = 24
PROF_CLASSES = ("gemm", "attn", "other", "lm_head", "sample", "fused")

EXPORTED = ["qw_config_default", "qw_init", "qw_destroy", "qw_kv_create", "qw_kv_destroy", "qw_kv_layout",
            "qw_prefill", "qw_decode_step", "qw_sample", "qw_check", "qw_last_error_message",
            "qw_debug_hidden", "qw_set_decode_path", "qw_debug_gemm", "qw_kernel_launches", "qw_attn_decode", "qw_attn_decode_noalloc", "qw_debug_trace",
            "qw_set_prefill_attention", "qw_generate", "qw_debug_profile", "qw_debug_inject_timeout"]


class QwConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("debug_hidden", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
                ("weight_bits", ctypes.c_int32)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class QwWeights(ctypes.Structure):
    _fields_ = [("embed_tokens", ctypes.c_void_p), ("norm", ctypes.c_void_p),
                ("input_layernorm", _PP), ("q_proj", _PP), ("k_proj", _PP), ("v_proj", _PP),
                ("q_norm", _PP), ("k_norm", _PP), ("o_proj", _PP), ("post_attention_layernorm", _PP),
                ("gate_proj", _PP), ("up_proj", _PP), ("down_proj", _PP), ("on_device", ctypes.c_int32)]


class QwSampleParams(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("reserved", ctypes.c_uint32), ("seed", ctypes.c_uint64)]


SAMPLE_PARAMS_BYTES = ctypes.sizeof(QwSampleParams)

_lib = None


class QwError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where} failed with {code}: {msg}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqwdecode.so (built by transformer_decode_qwen3_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.qw_config_default.argtypes = [ctypes.POINTER(QwConfig)]
    lib.qw_config_default.restype = None
    lib.qw_init.argtypes = [ctypes.POINTER(QwConfig), ctypes.POINTER(QwWeights), ctypes.POINTER(vp)]
    lib.qw_destroy.argtypes = [vp]
    lib.qw_kv_create.argtypes = [vp, i32, ctypes.POINTER(vp)]
    lib.qw_kv_destroy.argtypes = [vp]
    lib.qw_kv_layout.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i64),
                                 ctypes.POINTER(i32)]
    lib.qw_prefill.argtypes = [vp, vp, vp, ctypes.POINTER(i32), i32, vp, vp, i32, vp, vp]
    lib.qw_decode_step.argtypes = [vp, vp, vp, i32, vp, vp, i32, vp, vp]
    lib.qw_sample.argtypes = [vp, vp, i32, vp, ctypes.c_uint64, vp, vp]
    lib.qw_generate.argtypes = [vp, vp, vp, i32, vp, i32, i32, vp, ctypes.c_uint64, vp, vp]
    lib.qw_check.argtypes = [vp, vp]
    lib.qw_last_error_message.argtypes = []
    lib.qw_last_error_message.restype = ctypes.c_char_p
    lib.qw_debug_hidden.argtypes = [vp, i32, vp, i32, vp]
    lib.qw_set_decode_path.argtypes = [vp, i32]
    lib.qw_debug_gemm.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.qw_attn_decode.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, vp, vp]
    lib.qw_attn_decode_noalloc.argtypes = [vp, vp, i32, i32, i32, vp, i32, vp, i32, vp, vp]
    lib.qw_debug_trace.argtypes = [vp, i32, vp, i64, ctypes.POINTER(i64)]
    lib.qw_set_prefill_attention.argtypes = [vp, i32]
    lib.qw_debug_profile.argtypes = [vp, i32, vp, vp]
    lib.qw_debug_inject_timeout.argtypes = [vp]
    lib.qw_kernel_launches.argtypes = []
    lib.qw_kernel_launches.restype = ctypes.c_uint64
    for name in EXPORTED:
        if name not in ("qw_config_default", "qw_last_error_message", "qw_kernel_launches"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(rc: int, where: str):
    if rc != QW_OK:
        raise QwError(rc, where, _lib.qw_last_error_message().decode())


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def default_config(shape: ModelShape | None = None, max_batch: int = 64, max_tokens: int = 16384,
                   debug_hidden: bool = False, weight_bits: int = 16) -> QwConfig:
    lib = load()
    cfg = QwConfig()
    lib.qw_config_default(ctypes.byref(cfg))
    if shape is not None:
        cfg.n_layers, cfg.hidden, cfg.n_heads = shape.n_layers, shape.hidden, shape.n_heads
        cfg.n_kv_heads, cfg.head_dim, cfg.intermediate, cfg.vocab = (shape.n_kv_heads, shape.head_dim,
                                                                     shape.intermediate, shape.vocab)
    cfg.max_batch, cfg.max_tokens, cfg.debug_hidden = max_batch, max_tokens, int(debug_hidden)
    cfg.weight_bits = weight_bits
    return cfg


class Model:
    """A qw_ctx: weights uploaded from a name -> bf16 tensor dict (host or device)."""

    def __init__(self, weights: dict, shape: ModelShape, max_batch: int = 64, max_tokens: int = 16384,
                 debug_hidden: bool = False, weight_bits: int = 16):
        lib = load()
        self.shape = shape
        self.cfg = default_config(shape, max_batch, max_tokens, debug_hidden, weight_bits)
        L = shape.n_layers
        t0 = weights["model.embed_tokens.weight"]
        on_device = t0.is_cuda
        keep = []

        def p(t):
            assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.is_cuda == on_device
            keep.append(t)
            return t.data_ptr()

        def per_layer(suffix):
            arr = (ctypes.c_void_p * L)(*[p(weights[f"model.layers.{i}.{suffix}"]) for i in range(L)])
            keep.append(arr)
            return ctypes.cast(arr, _PP)

        w = QwWeights()
        w.embed_tokens = p(t0)
        w.norm = p(weights["model.norm.weight"])
        w.input_layernorm = per_layer("input_layernorm.weight")
        w.q_proj = per_layer("self_attn.q_proj.weight")
        w.k_proj = per_layer("self_attn.k_proj.weight")
        w.v_proj = per_layer("self_attn.v_proj.weight")
        w.q_norm = per_layer("self_attn.q_norm.weight")
        w.k_norm = per_layer("self_attn.k_norm.weight")
        w.o_proj = per_layer("self_attn.o_proj.weight")
        w.post_attention_layernorm = per_layer("post_attention_layernorm.weight")
        w.gate_proj = per_layer("mlp.gate_proj.weight")
        w.up_proj = per_layer("mlp.up_proj.weight")
        w.down_proj = per_layer("mlp.down_proj.weight")
        w.on_device = int(on_device)
        if on_device:
            torch.cuda.synchronize()
        h = ctypes.c_void_p()
        _check(lib.qw_init(ctypes.byref(self.cfg), ctypes.byref(w), ctypes.byref(h)), "qw_init")
        self.handle = h
        del keep

    def close(self):
        if getattr(self, "handle", None):
            _check(_lib.qw_destroy(self.handle), "qw_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_prefill_attention(self, variant: int):
        _check(_lib.qw_set_prefill_attention(self.handle, variant), "qw_set_prefill_attention")

    def set_decode_path(self, path: int):
        _check(_lib.qw_set_decode_path(self.handle, path), "qw_set_decode_path")

    def prefill(self, ids, positions, cu_seqlens, kv: "KVPool", block_tables, last_logits=None, stream=None):
        cu = [int(v) for v in cu_seqlens]
        cu_arr = (ctypes.c_int32 * len(cu))(*cu)
        _check(_lib.qw_prefill(self.handle, _ptr(ids), _ptr(positions), cu_arr, len(cu) - 1, kv.handle,
                               _ptr(block_tables), block_tables.shape[1], _ptr(last_logits), _stream(stream)),
               "qw_prefill")

    def decode_step(self, tokens, positions, kv: "KVPool", block_tables, logits=None, stream=None):
        _check(_lib.qw_decode_step(self.handle, _ptr(tokens), _ptr(positions), tokens.numel(), kv.handle,
                                   _ptr(block_tables), block_tables.shape[1], _ptr(logits), _stream(stream)),
               "qw_decode_step")

    def sample(self, params: torch.Tensor, rng_counter: int, out_ids, logits=None, batch=None, stream=None):
        batch = out_ids.numel() if batch is None else batch
        _check(_lib.qw_sample(self.handle, _ptr(logits), batch, _ptr(params), ctypes.c_uint64(rng_counter),
                              _ptr(out_ids), _stream(stream)), "qw_sample")

    def generate(self, first_token, start_pos: int, n_steps: int, params: torch.Tensor, rng_counter: int, out_ids,
                 kv: "KVPool", block_tables, stream=None):
        """n_steps decode + sample steps of one sequence with the ids fed back on the device."""
        _check(_lib.qw_generate(self.handle, kv.handle, _ptr(block_tables), block_tables.shape[-1], _ptr(first_token),
                                start_pos, n_steps, _ptr(params), ctypes.c_uint64(rng_counter), _ptr(out_ids),
                                _stream(stream)), "qw_generate")

    def attn_decode(self, q, positions, kv: "KVPool", layer: int, block_tables, out, stream=None):
        _check(_lib.qw_attn_decode(self.handle, _ptr(q), _ptr(positions), positions.numel(), kv.handle, layer,
                                   _ptr(block_tables), block_tables.shape[1], _ptr(out), _stream(stream)),
               "qw_attn_decode")

    def trace(self, enable: bool, fetch: bool = False):
        """Fused-decode phase stamps: returns a uint64 tensor [CTA, layers + 1, QW_TRACE_SLOTS] when fetch."""
        need = ctypes.c_int64()
        _check(_lib.qw_debug_trace(self.handle, int(enable), None, 0, ctypes.byref(need)), "qw_debug_trace")
        if not fetch:
            return None
        out = torch.zeros(need.value, dtype=torch.int64)
        _check(_lib.qw_debug_trace(self.handle, int(enable), out.data_ptr(), need.value, ctypes.byref(need)),
               "qw_debug_trace")
        return out.view(-1, self.shape.n_layers + 1, QW_TRACE_SLOTS)

    def profile(self, enable: bool, fetch: bool = False):
        """Per-kernel-class device time (qw_debug_profile): with fetch, a dict class -> (ms, launches)
        over the launches recorded since profiling was last enabled."""
        n = len(PROF_CLASSES)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        _check(_lib.qw_debug_profile(self.handle, int(enable), ctypes.addressof(ms) if fetch else None,
                                     ctypes.addressof(cnt) if fetch else None), "qw_debug_profile")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(PROF_CLASSES)} if fetch else None

    def inject_timeout(self):
        """Make the next fused decode step time out at one wait (failure-detection test hook)."""
        _check(_lib.qw_debug_inject_timeout(self.handle), "qw_debug_inject_timeout")

    def check(self, stream=None):
        _check(_lib.qw_check(self.handle, _stream(stream)), "qw_check")

    def check_code(self, stream=None) -> int:
        return _lib.qw_check(self.handle, _stream(stream))

    def debug_hidden(self, layer: int, out: torch.Tensor, n_rows: int, stream=None):
        _check(_lib.qw_debug_hidden(self.handle, layer, _ptr(out), n_rows, _stream(stream)), "qw_debug_hidden")


class KVPool:
    """A qw_kv paged cache: [n_layers][n_pages][2][n_kv][16][128] bf16."""

    def __init__(self, model: Model, n_pages: int):
        h = ctypes.c_void_p()
        _check(_lib.qw_kv_create(model.handle, n_pages, ctypes.byref(h)), "qw_kv_create")
        self.handle = h
        self.model = model
        base, ls, ps, npg = ctypes.c_void_p(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        _check(_lib.qw_kv_layout(h, ctypes.byref(base), ctypes.byref(ls), ctypes.byref(ps), ctypes.byref(npg)),
               "qw_kv_layout")
        self.base, self.layer_stride, self.page_stride, self.n_pages = base.value, ls.value, ps.value, npg.value

    def view(self) -> torch.Tensor:
        """The pool as a torch bf16 tensor [n_layers, n_pages, 2, n_kv, 16, 128] aliasing device memory."""
        S = self.model.shape
        shape = (S.n_layers, self.n_pages, 2, S.n_kv_heads, QW_PAGE_SIZE, QW_HEAD_DIM)
        n = 1
        for s in shape:
            n *= s
        return _tensor_from_ptr(self.base, n, torch.bfloat16).view(shape)

    def close(self):
        if getattr(self, "handle", None):
            _check(_lib.qw_kv_destroy(self.handle), "qw_kv_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _tensor_from_ptr(ptr: int, numel: int, dtype) -> torch.Tensor:
    """Wrap device memory owned by the library as a torch tensor (no copy, no ownership)."""
    class _Holder:
        def __init__(self):
            self.__cuda_array_interface__ = {"shape": (numel,), "typestr": "<u2" if dtype == torch.bfloat16 else "<f4",
                                             "data": (ptr, False), "version": 3}
    t = torch.as_tensor(_Holder(), device="cuda")
    return t.view(dtype) if dtype == torch.bfloat16 else t


def attn_decode_noalloc(q, positions, n_heads: int, n_kv_heads: int, kv_layer_ptr: int, n_pages: int,
                        block_tables, out, stream=None):
    """qw_attn_decode_noalloc: decode attention with the library's fixed scratch (no allocation)."""
    lib = load()
    _check(lib.qw_attn_decode_noalloc(_ptr(q), _ptr(positions), positions.numel(), n_heads, n_kv_heads, kv_layer_ptr,
                                      n_pages, _ptr(block_tables), block_tables.shape[1], _ptr(out), _stream(stream)),
           "qw_attn_decode_noalloc")


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load().qw_kernel_launches())


def debug_gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, epi: int = 0, bn: int = 256, split: int = 0,
               M: int | None = None, stream=None):
    """C (epilogue) = A B^T on the tensor-core projection kernel (see qw_debug_gemm).
    split = 1: A is the hi/lo layout and M the number of activation rows; split = 2: plain A on
    the CTA-pair (weight tile multicast) path."""
    lib = load()
    K = A.shape[1]
    M = A.shape[0] if M is None else M
    N = B.shape[0]
    _check(lib.qw_debug_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, epi, bn, int(split), _stream(stream)),
           "qw_debug_gemm")


def sample_params(rows: list[tuple[float, int, float, int]], device="cuda") -> torch.Tensor:
    """Pack (temperature, top_k, top_p, seed) rows into a device qw_sample_params array."""
    arr = (QwSampleParams * len(rows))()
    for i, (t, k, p, s) in enumerate(rows):
        arr[i].temperature, arr[i].top_k, arr[i].top_p, arr[i].reserved, arr[i].seed = t, k, p, 0, s
    raw = bytes(arr)
    host = torch.frombuffer(bytearray(raw), dtype=torch.uint8)
    return host.to(device)
