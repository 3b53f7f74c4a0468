"""ctypes wrapper of the plain single-precision C oracle (oracle/qwen3_ref.c).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the benchmark's CPU
baseline, never by the product path.  It shares no code with the CUDA library; the
weights and caches it reads come from the seeded input generator.

build() compiles qwen3_ref.c with gcc (OpenMP, -O2) into liboracle_qwen3.so next to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qwen3_ref.c")
LIB = os.path.join(HERE, "liboracle_qwen3.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle if needed (portable C: no architecture flags)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", LIB, SRC, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stdout + r.stderr)
    return LIB


_PP = ctypes.POINTER(ctypes.c_void_p)


class _Model(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("eps", ctypes.c_float), ("theta", ctypes.c_double),
                ("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("in_norm", _PP), ("wq", _PP), ("wk", _PP), ("wv", _PP), ("q_norm", _PP), ("k_norm", _PP),
                ("wo", _PP), ("post_norm", _PP), ("wg", _PP), ("wu", _PP), ("wd", _PP)]


class _Cache(ctypes.Structure):
    _fields_ = [("cap", ctypes.c_int32), ("len", ctypes.c_int32), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("pos", ctypes.c_void_p)]


class _SampleInfo(ctypes.Structure):
    _fields_ = [("id", ctypes.c_int32), ("cutoff", ctypes.c_int32), ("cum_at_cutoff", ctypes.c_double),
                ("cum_before_cutoff", ctypes.c_double), ("draw_gap", ctypes.c_double)]


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        lib.qwo_forward.argtypes = [ctypes.POINTER(_Model), vp, vp, i32, ctypes.POINTER(_Cache), i32, vp, vp]
        lib.qwo_sample.argtypes = [vp, i32, ctypes.c_float, i32, ctypes.c_float, ctypes.c_double,
                                   ctypes.POINTER(_SampleInfo)]
        lib.qwo_sampling_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.qwo_sampling_uniform.restype = ctypes.c_double
        lib.qwo_philox4x32_10.argtypes = [vp, vp, vp]
        lib.qwo_rms_norm.argtypes = [vp, vp, i32, ctypes.c_float, vp]
        lib.qwo_rope.argtypes = [vp, i32, i32, ctypes.c_double]
        lib.qwo_generate.argtypes = [ctypes.POINTER(_Model), vp, i32, i32, ctypes.c_float, i32, ctypes.c_float,
                                     ctypes.c_uint64, ctypes.POINTER(_Cache), vp, vp]
        lib.qwo_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _bits(t) -> np.ndarray:
    """bf16 values (torch.bfloat16 tensor) as a contiguous uint16 numpy array."""
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


class Cache:
    """One sequence's cache for the C oracle: float32 K and V [n_layers][n_kv][cap][head_dim]."""

    def __init__(self, shape, cap: int):
        self.cap = cap
        self.k = np.zeros((shape.n_layers, shape.n_kv_heads, cap, shape.head_dim), dtype=np.float32)
        self.v = np.zeros_like(self.k)
        self.pos = np.zeros(cap, dtype=np.int32)
        self.c = _Cache(cap, 0, _p(self.k), _p(self.v), _p(self.pos))

    @property
    def len(self) -> int:
        return self.c.len

    def fill_prefix(self, layer: int, k, v):
        """Entries 0..L-1 of one layer from [L, n_kv, head_dim] arrays (positions 0..L-1); call for every
        layer, then set_len(L)."""
        L = k.shape[0]
        self.k[layer, :, :L] = np.asarray(k, dtype=np.float32).transpose(1, 0, 2)
        self.v[layer, :, :L] = np.asarray(v, dtype=np.float32).transpose(1, 0, 2)
        self.pos[:L] = np.arange(L, dtype=np.int32)

    def set_len(self, L: int):
        self.c.len = L


class COracle:
    """Steps 2-9 of the article in plain C: weights are the generator's bf16 tensors."""

    def __init__(self, weights: dict, shape, eps: float = 1e-6, theta: float = 1e6):
        lib = load()
        self.shape = shape
        L = shape.n_layers
        self._keep = {k: _bits(v) for k, v in weights.items()}
        m = _Model()
        m.n_layers, m.hidden, m.n_heads, m.n_kv_heads = L, shape.hidden, shape.n_heads, shape.n_kv_heads
        m.head_dim, m.intermediate, m.vocab, m.eps, m.theta = (shape.head_dim, shape.intermediate, shape.vocab, eps,
                                                               theta)
        m.embed = _p(self._keep["model.embed_tokens.weight"])
        m.final_norm = _p(self._keep["model.norm.weight"])
        self._arrays = []

        def per_layer(suffix):
            arr = (ctypes.c_void_p * L)(*[_p(self._keep[f"model.layers.{i}.{suffix}"]) for i in range(L)])
            self._arrays.append(arr)
            return ctypes.cast(arr, _PP)

        m.in_norm = per_layer("input_layernorm.weight")
        m.wq, m.wk, m.wv = (per_layer(f"self_attn.{n}_proj.weight") for n in "qkv")
        m.q_norm, m.k_norm = per_layer("self_attn.q_norm.weight"), per_layer("self_attn.k_norm.weight")
        m.wo = per_layer("self_attn.o_proj.weight")
        m.post_norm = per_layer("post_attention_layernorm.weight")
        m.wg, m.wu, m.wd = (per_layer(f"mlp.{n}_proj.weight") for n in ("gate", "up", "down"))
        self.m = m
        self.lib = lib

    def new_cache(self, cap: int) -> Cache:
        return Cache(self.shape, cap)

    def forward(self, ids, positions, cache: Cache, last_only: bool = False, hiddens: bool = False):
        """Logits [T, vocab] ([1, vocab] with last_only) as float32; with hiddens also the residual
        stream after every block, [n_layers, T, hidden]."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        T = ids.size
        S = self.shape
        logits = np.empty((1 if last_only else T, S.vocab), dtype=np.float32)
        hid = np.empty((S.n_layers, T, S.hidden), dtype=np.float32) if hiddens else None
        rc = self.lib.qwo_forward(ctypes.byref(self.m), _p(ids), _p(pos), T, ctypes.byref(cache.c), int(last_only),
                                  _p(logits), _p(hid) if hid is not None else None)
        if rc:
            raise RuntimeError(f"qwo_forward failed with {rc}")
        return (logits, hid) if hiddens else logits

    def generate(self, prompt_ids, n_steps: int, temperature=0.0, top_k=0, top_p=1.0, seed=0):
        """Step 9 loop; (ids [n_steps], logits rows [n_steps, vocab])."""
        prompt = np.ascontiguousarray(prompt_ids, dtype=np.int32)
        cache = self.new_cache(prompt.size + n_steps)
        out = np.empty(n_steps, dtype=np.int32)
        rows = np.empty((n_steps, self.shape.vocab), dtype=np.float32)
        rc = self.lib.qwo_generate(ctypes.byref(self.m), _p(prompt), prompt.size, n_steps, temperature, top_k, top_p,
                                   seed, ctypes.byref(cache.c), _p(out), _p(rows))
        if rc:
            raise RuntimeError(f"qwo_generate failed with {rc}")
        return out.tolist(), rows


def sample_detail(logits, temperature: float, top_k: int, top_p: float, u: float) -> dict:
    """qwo_sample on one float32 logits row, with the quantities the near-tie exemptions need."""
    lib = load()
    row = np.ascontiguousarray(logits, dtype=np.float32)
    info = _SampleInfo()
    rc = lib.qwo_sample(_p(row), row.size, temperature, top_k, top_p, u, ctypes.byref(info))
    if rc < 0:
        raise RuntimeError(f"qwo_sample failed with {rc}")
    return {"id": info.id, "cutoff": info.cutoff or None, "cum_at_cutoff": info.cum_at_cutoff,
            "cum_before_cutoff": info.cum_before_cutoff, "draw_gap": info.draw_gap, "u": u}


def sampling_uniform(seed: int, rng_counter: int) -> float:
    return load().qwo_sampling_uniform(seed, rng_counter)


def philox4x32_10(ctr, key):
    c = np.array(ctr, dtype=np.uint32)
    k = np.array(key, dtype=np.uint32)
    out = np.empty(4, dtype=np.uint32)
    load().qwo_philox4x32_10(_p(c), _p(k), _p(out))
    return tuple(int(v) for v in out)


def rms_norm(x, w_bf16) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = _bits(w_bf16)
    y = np.empty_like(x)
    load().qwo_rms_norm(_p(x), _p(w), x.size, 1e-6, _p(y))
    return y


def rope(x, pos: int, theta: float = 1e6) -> np.ndarray:
    y = np.array(x, dtype=np.float32)
    load().qwo_rope(_p(y), y.size, pos, theta)
    return y


def threads() -> int:
    return load().qwo_threads()
