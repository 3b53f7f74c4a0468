"""Benchmark of the Qwen3-0.6B-shaped decoder pass on one GB300.

Workloads (--workload; the default is the headline):
  decode_bs1       batch-1 greedy decode after a 512-token random prompt; the timed steps
                   run at cache positions 512 .. 512 + K - 1 (K = 256 covers 512 -> 768).
                   One step = embedding, 28 blocks, final norm, tied LM head and the
                   greedy sampler, the sampled id fed back on the device.
  decode_bs64      64 sequences over ragged synthetic caches of 128..4096 positions
                   (16-token pages), one decode step + sampling (T 0.7, top-k 50,
                   top-p 0.9, Philox seeded by sequence id) per timed step.
  prefill          prefill of 8 x 2048 random tokens (causal), last-token logits.
  decode_bs16_32k  16 sequences at cache length 32768 (synthetic caches, ~60 GB of
                   bf16 KV), greedy decode steps at positions 32768 .. 32768 + K - 1.
  decode_bs1_int8  decode_bs1 with weight-only int8 weights (one power-of-two scale per
                   output channel): the fused batch-1 kernel streams the int8 codes.
The other workloads are also measured briefly and reported under "secondary".

Random-init weights (seeded, N(0, 0.02)-shaped) and random token ids: no dataset,
no checkpoint.  Every step streams 1.19 GB of weights (and up to 60 GB of cache),
more than the 129 MB L2, so no flush is needed between steps.

The library is single-GPU: it runs on the current CUDA device only and this
script measures one GPU.  Asked for more (--gpus N > 1, or a torchrun launch
with WORLD_SIZE > 1), rank 0 prints one line saying so and nothing runs.

--impl reference times the plain single-precision C oracle (OpenMP over the host
cores) on a bounded sample of the same workload, with the same metric and config.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from transformer_decode_qwen3_gb300 import synth  # noqa: E402

S = synth.QWEN3_0_6B
PAGE = 16
LAYER_PARAMS = (S.n_heads * S.head_dim * S.hidden + 2 * S.n_kv_heads * S.head_dim * S.hidden +
                S.hidden * S.n_heads * S.head_dim + 3 * S.intermediate * S.hidden)
NORM_BYTES = 2 * (2 * S.hidden + 2 * S.head_dim)
WEIGHT_BYTES = S.n_layers * (2 * LAYER_PARAMS + NORM_BYTES) + 2 * S.hidden + 2 * S.vocab * S.hidden
# int8 codes + one fp32 scale per output channel (q|k|v rows, o_proj rows, gate/up rows, down rows)
SCALES_PER_LAYER = (S.n_heads + 2 * S.n_kv_heads) * S.head_dim + S.hidden + 2 * S.intermediate + S.hidden
WEIGHT_BYTES_INT8 = (S.n_layers * (LAYER_PARAMS + 4 * SCALES_PER_LAYER + NORM_BYTES) + 2 * S.hidden +
                     S.vocab * S.hidden + 4 * S.vocab)
KV_BYTES_PER_POS = S.n_layers * 2 * S.n_kv_heads * S.head_dim * 2          # 114,688 B per cached position
KV_LAYER_BYTES_PER_POS = KV_BYTES_PER_POS // S.n_layers                     # 4,096 B
PROMPT, PREFILL_B, PREFILL_T, BS64, LONG_B, LONG_L = 512, 8, 2048, 64, 16, 32768
METRICS = {
    "decode_bs1": "decode tok/s @bs1 (Qwen3-0.6B shape, 512-token prompt, greedy)",
    "decode_bs64": "decode tok/s @bs64 (Qwen3-0.6B shape, ragged caches 128..4096, sampled)",
    "prefill": "prefill tok/s (Qwen3-0.6B shape, 8 x 2048 causal)",
    "decode_bs16_32k": "decode tok/s @bs16 (Qwen3-0.6B shape, caches at 32768, greedy)",
    "decode_bs1_int8": "decode tok/s @bs1 (Qwen3-0.6B shape, weight-only int8, 512-token prompt, greedy)",
}


def config_of(name: str, K: int) -> dict:
    """The workload description both arms print (no model keys: the shape is in the metric)."""
    l2 = "inputs larger than L2 (1.19 GB of weights streamed per step), no flush"
    if name in ("decode_bs1", "decode_bs1_int8"):
        q8 = name == "decode_bs1_int8"
        return {"workload": f"decode bs1, prompt {PROMPT}, timed cache positions {PROMPT}..{PROMPT + K - 1}, greedy"
                            + (", weight-only int8 per output channel" if q8 else ""),
                "global_batch": 1, "prompt": PROMPT, "cache_start": PROMPT, "cache_end": PROMPT + K,
                "weights": "int8 codes + fp32 scale per output channel" if q8 else "bf16", "l2": l2}
    if name == "decode_bs64":
        return {"workload": "decode bs64, ragged paged caches 128..4096, T 0.7 / top-k 50 / top-p 0.9",
                "global_batch": BS64, "page": PAGE, "l2": l2}
    if name == "prefill":
        return {"workload": f"prefill {PREFILL_B} x {PREFILL_T}, causal GQA", "global_batch": PREFILL_B,
                "seq_len": PREFILL_T, "l2": l2}
    return {"workload": f"decode bs{LONG_B}, caches at {LONG_L}, timed positions {LONG_L}..{LONG_L + K - 1}, greedy",
            "global_batch": LONG_B, "cache_start": LONG_L, "cache_end": LONG_L + K, "page": PAGE, "l2": l2}


# DRAM bytes (read + write) of each workload's roofline kernel, from one ncu capture summarised
# under profiles/ (per launch of the fused kernel; per step for the 28 attention launches of a
# decode batch, like the algorithmic bytes they are compared with); reported only while the
# kernel's source file is the one that was captured (its sha256 below), else null.
NCU_TRAFFIC = {
    "decode_bs1": ("transformer_decode_qwen3_gb300/csrc/qw_fused.cu",
                   "a83d5ec64dd7d9023de2bdccd5f24dd80b1e1c80d177932f8f4d7700ea76845c", 1266.07e6),
    "decode_bs1_int8": ("transformer_decode_qwen3_gb300/csrc/qw_fused.cu",
                        "a83d5ec64dd7d9023de2bdccd5f24dd80b1e1c80d177932f8f4d7700ea76845c", 667.93e6),
    # all 28 layers of a step: split-KV attention (552.41 MB) + merge (3.02 MB) per layer
    "decode_bs64": ("transformer_decode_qwen3_gb300/csrc/qw_kernels.cu",
                    "9802f1b4fabf1b2e6302f2fce2bd189570c40b04cdcda5c7e94c74070000ad3d", 28 * (552.41e6 + 3.02e6)),
}


def ncu_traffic(name):
    ent = NCU_TRAFFIC.get(name)
    if ent is None:
        return None
    path, sha, nbytes = ent
    with open(os.path.join(ROOT, path), "rb") as f:
        return nbytes if hashlib.sha256(f.read()).hexdigest() == sha else None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [t.strip() for t in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        busy = [v for v in sm if mx is None or v > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def timed(fn, K):
    """Run fn(i) for i < K between synchronizes; CUDA-event milliseconds and kernel launches."""
    from transformer_decode_qwen3_gb300 import binding as bd
    torch.cuda.synchronize()
    launches0 = bd.kernel_launches()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for i in range(K):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), bd.kernel_launches() - launches0


def profiled(model, fn, K):
    """Per-kernel-class device milliseconds per step over K more steps (library CUDA events)."""
    torch.cuda.synchronize()
    model.profile(True)
    for i in range(K):
        fn(i)
    prof = model.profile(False, fetch=True)
    return {k: {"ms_per_step": v[0] / K, "launches_per_step": v[1] / K} for k, v in prof.items() if v[1]}


# ------------------------------------------------------------------ workloads
def synth_caches(bd, model, lens, cap):
    """A KV pool holding the synthetic caches of sequences with lengths `lens` (room for `cap`
    positions each), pages assigned in order; returns (pool, block tables)."""
    per = math.ceil(cap / PAGE) + 1
    kv = bd.KVPool(model, len(lens) * per)
    pool = kv.view()
    bt = torch.arange(len(lens) * per, dtype=torch.int32, device="cuda").view(len(lens), per)
    for s, L in enumerate(lens):
        n_p = math.ceil(L / PAGE)
        for layer in range(S.n_layers):
            for which, std in ((0, 1.0), (1, 0.64)):
                v = synth.kv_values(0, layer, which, s * (1 << 15) * 1024, L * 1024, std, "cuda")
                if n_p * PAGE > L:
                    v = torch.cat([v.view(L, 8, 128), torch.zeros(n_p * PAGE - L, 8, 128, dtype=torch.bfloat16,
                                                                  device="cuda")])
                pool[layer, s * per:s * per + n_p, which] = v.view(n_p, PAGE, 8, 128).permute(0, 2, 1, 3)
    return kv, bt


class DecodeBs1:
    """Batch 1: a prompt of 512 random ids, then greedy decode steps."""
    units_per_step = 1
    roofline_class = "fused"

    def __init__(self, bd, model, n_steps):
        self.bd, self.model = bd, model
        self.n_pages = math.ceil((PROMPT + n_steps + 1) / PAGE) + 1
        self.kv = bd.KVPool(model, self.n_pages)
        self.bt = torch.arange(self.n_pages, dtype=torch.int32, device="cuda").view(1, -1)
        ids = synth.token_ids(0, 1, PROMPT, S.vocab, device="cuda")
        model.prefill(ids, torch.arange(PROMPT, dtype=torch.int32, device="cuda"), [0, PROMPT], self.kv, self.bt,
                      None)
        self.params = bd.sample_params([(0.0, 1, 1.0, 0)])
        self.toks = torch.empty(n_steps + 1, dtype=torch.int32, device="cuda")
        self.pos = torch.arange(PROMPT, PROMPT + n_steps, dtype=torch.int32, device="cuda")
        model.sample(self.params, 0, self.toks[0:1])
        model.check()

    def step(self, i):
        self.model.decode_step(self.toks[i:i + 1], self.pos[i:i + 1], self.kv, self.bt, None)
        self.model.sample(self.params, i + 1, self.toks[i + 1:i + 2])

    def bytes_per_step(self, K):
        return WEIGHT_BYTES + sum((PROMPT + i + 1) * KV_BYTES_PER_POS for i in range(K)) / K

    def roofline_bytes(self, K):
        return self.bytes_per_step(K)

    def e2e(self, K):
        """Token and position from pinned host memory in, sampled id out, every step."""
        h_tok = torch.empty(1, dtype=torch.int32).pin_memory()
        h_pos = torch.empty(1, dtype=torch.int32).pin_memory()
        h_out = torch.empty(1, dtype=torch.int32).pin_memory()
        d_tok = torch.empty(1, dtype=torch.int32, device="cuda")
        d_pos = torch.empty(1, dtype=torch.int32, device="cuda")
        d_out = torch.empty(1, dtype=torch.int32, device="cuda")
        h_tok[0] = int(self.toks[0])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(K):
            h_pos[0] = PROMPT + i
            d_tok.copy_(h_tok, non_blocking=True)
            d_pos.copy_(h_pos, non_blocking=True)
            self.model.decode_step(d_tok, d_pos, self.kv, self.bt, None)
            self.model.sample(self.params, i + 1, d_out)
            h_out.copy_(d_out, non_blocking=True)
            torch.cuda.current_stream().synchronize()
            h_tok[0] = int(h_out[0])
        return time.perf_counter() - t0, 8, 4

    def generate_e2e(self, K):
        """qw_generate: the first token in from pinned host memory, K steps decoded, sampled and fed
        back on the device, the K ids out to the host; wall-clock seconds."""
        h_tok = torch.empty(1, dtype=torch.int32).pin_memory()
        h_out = torch.empty(K, dtype=torch.int32).pin_memory()
        d_tok = torch.empty(1, dtype=torch.int32, device="cuda")
        d_out = torch.empty(K, dtype=torch.int32, device="cuda")
        h_tok[0] = int(self.toks[0])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        d_tok.copy_(h_tok, non_blocking=True)
        self.model.generate(d_tok, PROMPT, K, self.params, 1, d_out, self.kv, self.bt)
        h_out.copy_(d_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return time.perf_counter() - t0

    def close(self):
        self.kv.close()


class DecodeBs1Int8(DecodeBs1):
    """DecodeBs1 on the weight-only int8 model: the fused kernel streams 0.60 GB of codes a step."""

    def bytes_per_step(self, K):
        return WEIGHT_BYTES_INT8 + sum((PROMPT + i + 1) * KV_BYTES_PER_POS for i in range(K)) / K


class BatchDecode:
    """Batched decode over synthetic paged caches, one step per sequence per timed step."""
    roofline_class = "attn"

    def __init__(self, bd, model, lens, params, cap):
        self.bd, self.model = bd, model
        self.lens = lens
        self.B = len(lens)
        self.units_per_step = self.B
        self.kv, self.bt = synth_caches(bd, model, lens, cap)
        self.toks = synth.token_ids(0, 3, self.B, S.vocab, device="cuda")
        self.base = torch.tensor(lens, dtype=torch.int32, device="cuda")
        self.params = bd.sample_params(params)
        self.out = torch.empty(self.B, dtype=torch.int32, device="cuda")

    def positions(self, i):
        return self.base

    def step(self, i):
        self.model.decode_step(self.toks, self.positions(i), self.kv, self.bt, None)
        self.model.sample(self.params, i, self.out)

    def attention_bytes(self, i=0):
        return sum((L + 1) * KV_LAYER_BYTES_PER_POS for L in self.lens) * S.n_layers

    def bytes_per_step(self, K=1):
        return WEIGHT_BYTES + self.attention_bytes()

    def roofline_bytes(self, K):
        return self.attention_bytes()

    def e2e(self, K):
        """Tokens and positions from pinned host memory in, sampled ids out, every step."""
        h_in = torch.empty(K, 2, self.B, dtype=torch.int32).pin_memory()
        for i in range(K):
            h_in[i, 0] = self.toks.cpu()
            h_in[i, 1] = self.positions(i).cpu()
        h_out = torch.empty(self.B, dtype=torch.int32).pin_memory()
        d_in = torch.empty(2, self.B, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(K):
            d_in.copy_(h_in[i], non_blocking=True)
            self.model.decode_step(d_in[0], d_in[1], self.kv, self.bt, None)
            self.model.sample(self.params, i, self.out)
            h_out.copy_(self.out, non_blocking=True)
            torch.cuda.current_stream().synchronize()
        return time.perf_counter() - t0, 2 * self.B * 4, self.B * 4

    def close(self):
        self.kv.close()


class DecodeBs64(BatchDecode):
    """Batch 64: ragged synthetic caches 128..4096, one sampled step each (the same step repeated)."""

    def __init__(self, bd, model, K):
        lens = synth.uniform_ints(0, synth.STREAM_LENGTHS, BS64, 128, 4096).tolist()
        super().__init__(bd, model, lens, [(0.7, 50, 0.9, s) for s in range(BS64)], 4096 + PAGE)


class DecodeBs16Long(BatchDecode):
    """Batch 16 at cache length 32768: greedy steps at positions 32768 + i (the cache grows)."""

    def __init__(self, bd, model, K):
        super().__init__(bd, model, [LONG_L] * LONG_B, [(0.0, 1, 1.0, s) for s in range(LONG_B)], LONG_L + K + 8)
        self.K = K
        self.pos = self.base.view(1, -1) + torch.arange(K + 8, dtype=torch.int32, device="cuda").view(-1, 1)

    def positions(self, i):
        return self.pos[i % (self.K + 8)]

    def attention_bytes(self, i=None):
        return self.B * (LONG_L + 1 + (self.K - 1) / 2) * KV_LAYER_BYTES_PER_POS * S.n_layers


class Prefill:
    """Prefill only: 8 x 2048 random prompts, last-token logits."""
    units_per_step = PREFILL_B * PREFILL_T
    roofline_class = "gemm"

    def __init__(self, bd, model, K):
        self.bd, self.model = bd, model
        B, T = PREFILL_B, PREFILL_T
        self.kv = bd.KVPool(model, B * T // PAGE)
        self.bt = torch.arange(B * T // PAGE, dtype=torch.int32, device="cuda").view(B, -1)
        self.ids = synth.token_ids(0, 2, B * T, S.vocab, device="cuda")
        self.pos = torch.arange(T, dtype=torch.int32, device="cuda").repeat(B)
        self.cu = [T * s for s in range(B + 1)]
        self.last = torch.empty(B, S.vocab, device="cuda")
        self.params = bd.sample_params([(0.0, 1, 1.0, s) for s in range(B)])
        self.out = torch.empty(B, dtype=torch.int32, device="cuda")

    def step(self, i):
        self.model.prefill(self.ids, self.pos, self.cu, self.kv, self.bt, self.last)

    def flops(self):
        B, T = PREFILL_B, PREFILL_T
        linear = 2 * LAYER_PARAMS * S.n_layers * B * T
        attn = 2 * S.n_heads * S.head_dim * T * T * S.n_layers * B      # causal: half of 4 H d T^2
        head = 2 * S.hidden * S.vocab * B
        return linear, attn, head

    def e2e(self, K):
        B, T = PREFILL_B, PREFILL_T
        h_in = torch.empty(2, B * T, dtype=torch.int32).pin_memory()
        h_in[0] = self.ids.cpu()
        h_in[1] = self.pos.cpu()
        h_out = torch.empty(B, dtype=torch.int32).pin_memory()
        d_in = torch.empty(2, B * T, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(K):
            d_in.copy_(h_in, non_blocking=True)
            self.model.prefill(d_in[0], d_in[1], self.cu, self.kv, self.bt, self.last)
            self.model.sample(self.params, 0, self.out, logits=self.last)
            h_out.copy_(self.out, non_blocking=True)
            torch.cuda.current_stream().synchronize()
        return time.perf_counter() - t0, 2 * B * T * 4, B * 4

    def close(self):
        self.kv.close()


# ------------------------------------------------------------------ CPU oracle
def oracle_rate(workload: str, max_seconds=15.0):
    """The C oracle (plain single precision, OpenMP over the host cores), unmodified, on a bounded
    sample of the workload; (units/s, sample text, threads)."""
    import numpy as np
    from oracle import qwen3_c as C
    w = synth.make_weights(S)
    if workload == "decode_bs1_int8":
        # the oracle's own quantiser; the dequantised weights are exactly bf16 values
        from oracle import qwen3_ref as R
        for k in list(w):
            if k == "model.embed_tokens.weight" or k.endswith(R.QUANTISED_SUFFIXES):
                deq = R.dequantize_rows_int8(*R.quantize_rows_int8(w[k]))
                w[k] = torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16)
    orc = C.COracle(w, S)
    threads = C.threads()
    if workload == "prefill":
        T = 128                         # a 128-token prefix of sequence 0
        ids = synth.token_ids(0, 2, T, S.vocab).numpy()
        t0 = time.perf_counter()
        orc.forward(ids, np.arange(T), orc.new_cache(T), last_only=True)
        dt = time.perf_counter() - t0
        return T / dt, f"prefill of the first {T} tokens of one 2048-token sequence ({dt:.1f} s)", threads
    if workload in ("decode_bs64", "decode_bs16_32k"):
        if workload == "decode_bs64":
            lens = synth.uniform_ints(0, synth.STREAM_LENGTHS, BS64, 128, 4096).tolist()
            params = (0.7, 50, 0.9)
        else:
            lens = [LONG_L] * LONG_B
            params = (0.0, 1, 1.0)
        toks = synth.token_ids(0, 3, len(lens), S.vocab)
        per_tok = S.n_kv_heads * 128
        elapsed, n = 0.0, 0
        while n < 1 or (elapsed < max_seconds and n < len(lens)):
            L = lens[n]
            cache = orc.new_cache(L + 1)
            for layer in range(S.n_layers):        # cache set-up, not timed
                k = synth.kv_values(0, layer, 0, n * (1 << 15) * per_tok, L * per_tok, 1.0)
                v = synth.kv_values(0, layer, 1, n * (1 << 15) * per_tok, L * per_tok, 0.64)
                cache.fill_prefix(layer, synth.bf16_to_f32(k).numpy().reshape(L, 8, 128),
                                  synth.bf16_to_f32(v).numpy().reshape(L, 8, 128))
            cache.set_len(L)
            t0 = time.perf_counter()
            logits = orc.forward([int(toks[n])], [L], cache, last_only=True)
            C.sample_detail(logits[0], *params, C.sampling_uniform(n, 0))
            elapsed += time.perf_counter() - t0
            n += 1
            del cache
        return n / elapsed, (f"{n} of the {len(lens)} sequences, one decode step each ({elapsed:.1f} s timed; "
                             f"cache set-up untimed)"), threads
    ids = synth.token_ids(0, 1, PROMPT, S.vocab).numpy()
    cache = orc.new_cache(PROMPT + 4096)
    logits = orc.forward(ids, np.arange(PROMPT), cache, last_only=True)
    tok = int(np.argmax(logits[0]))
    t0 = time.perf_counter()
    n = 0
    while n < 2 or (time.perf_counter() - t0 < max_seconds and n < 4096):
        logits = orc.forward([tok], [PROMPT + n], cache, last_only=True)
        tok = int(np.argmax(logits[0]))
        n += 1
    dt = time.perf_counter() - t0
    return n / dt, f"{n} batch-1 greedy decode steps after the 512-token prompt ({dt:.1f} s; prefill untimed)", threads


def run_reference(args):
    v, sample, threads = oracle_rate(args.workload, max_seconds=max(5.0, min(60.0, 0.25 * args.steps)))
    unit = "tok/s"
    line = {"metric": METRICS[args.workload], "value": v, "unit": unit, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded random-init weights and token ids)",
            "impl": "reference", "config": config_of(args.workload, args.steps),
            "cpu_baseline": {"value": v, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main
def make_workload(name, bd, model, K, W):
    if name == "decode_bs1":
        return DecodeBs1(bd, model, max(K, W))
    if name == "decode_bs1_int8":
        return DecodeBs1Int8(bd, model, max(K, W))
    if name == "decode_bs64":
        return DecodeBs64(bd, model, max(K, W))
    if name == "decode_bs16_32k":
        return DecodeBs16Long(bd, model, max(K, W))
    return Prefill(bd, model, max(K, W))


def measure(name, bd, model, K, W, hbm, tf_burst):
    """Returns the JSON fields of one workload measured with K timed steps after W warm-ups."""
    wl = make_workload(name, bd, model, K, W)
    for i in range(W):
        wl.step(i)
    ms, launches = timed(wl.step, K)
    out = {"ms_per_step": ms / K, "value": wl.units_per_step * K / (ms / 1e3), "gpu_launches": launches}
    # per-kernel-class device time over K more steps, CUDA events on the launching stream
    kern = profiled(model, wl.step, K)
    out["kernels"] = kern
    cls_ms = kern.get(wl.roofline_class, {}).get("ms_per_step")
    if name == "prefill":
        lin, attn, head = wl.flops()
        ach = lin / (cls_ms / 1e3) / 1e12
        attn_ms = kern["attn"]["ms_per_step"]
        out["roofline"] = {"bound": "tensor", "kernel": "prefill projections (tcgen05 GEMMs, all 4 x 28 per step)",
                           "achieved": ach, "peak": tf_burst, "unit": "TFLOP/s", "frac": ach / tf_burst,
                           "traffic": None, "algorithmic_flop": lin, "kernel_ms": cls_ms,
                           "gemm_frac": ach / tf_burst,
                           "attention_frac": attn / (attn_ms / 1e3) / 1e12 / tf_burst,
                           "step_frac": (lin + attn + head) / (ms / K / 1e3) / 1e12 / tf_burst}
    else:
        nbytes = wl.roofline_bytes(K)
        ach = nbytes / (cls_ms / 1e3) / 1e9
        what = {"decode_bs1": "decode step (the fused batch-1 kernel)",
                "decode_bs1_int8": "decode step (the fused batch-1 kernel streaming int8 weights)"}.get(
                    name, "split-KV decode attention + merge (all 28 layers of a step)")
        out["roofline"] = {"bound": "hbm", "kernel": what, "achieved": ach, "peak": hbm, "unit": "GB/s",
                           "frac": ach / hbm, "traffic": ncu_traffic(name), "algorithmic_bytes": nbytes,
                           "kernel_ms": cls_ms,
                           "step_hbm_frac": wl.bytes_per_step(K) / (ms / K / 1e3) / 1e9 / hbm}
    e2e_s, h2d, d2h = wl.e2e(K)
    out["e2e"] = {"value": wl.units_per_step * K / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h}
    if name == "decode_bs1":  # the whole loop on the device (qw_generate), host copies at the ends only
        out["generate"] = {"value": K / wl.generate_e2e(K), "unit": "tok/s", "h2d_bytes": 4, "d2h_bytes": 4 * K}
    wl.close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--workload", default="decode_bs1", choices=list(METRICS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 or world > 1:
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps({"metric": METRICS[args.workload], "impl": args.impl, "n_gpus": max(args.gpus, world),
                              "unavailable": "single-GPU library: it measures one GPU only"}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    from transformer_decode_qwen3_gb300 import binding as bd
    bd.load()
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    w = synth.make_weights(S, device="cuda")             # bit-identical to the CPU generator
    model = bd.Model(w, S, max_batch=64, max_tokens=PREFILL_B * PREFILL_T)
    del w
    torch.cuda.empty_cache()
    models = {"bf16": model}

    def model_for(name):
        """The int8 workload runs on its own context (weights quantised at qw_init)."""
        if name != "decode_bs1_int8":
            return models["bf16"]
        if "int8" not in models:
            w8 = synth.make_weights(S, device="cuda")
            models["int8"] = bd.Model(w8, S, max_batch=8, max_tokens=1024, weight_bits=8)
            del w8
            torch.cuda.empty_cache()
        return models["int8"]

    with ClockSampler(torch.cuda.current_device()) as clk:
        m = measure(args.workload, bd, model_for(args.workload), args.steps, args.warmup, hbm, tf_burst)
    m["roofline"]["peak_kind"] = f"{peak_kind} ({'copy bandwidth' if m['roofline']['unit'] == 'GB/s' else 'bf16 burst'})"
    line = {"metric": METRICS[args.workload], "value": m["value"], "unit": "tok/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random-init bf16 weights and token ids)",
            "config": config_of(args.workload, args.steps), "roofline": m["roofline"], "e2e": m["e2e"],
            "gpu_launches": m["gpu_launches"], "kernels": m["kernels"], "clocks": clk.summary()}
    if "generate" in m:
        line["generate"] = m["generate"]
    if not args.no_secondary:
        sec = {}
        for name in METRICS:
            if name == args.workload:
                continue
            K2 = 64 if name in ("decode_bs1", "decode_bs1_int8") else (16 if name == "decode_bs16_32k" else 5)
            r = measure(name, bd, model_for(name), K2, 3, hbm, tf_burst)
            sec[name] = {"tok_s": r["value"], "ms_per_step": r["ms_per_step"], "roofline": r["roofline"],
                         "e2e_tok_s": r["e2e"]["value"], "kernels": r["kernels"], "config": config_of(name, K2)}
            torch.cuda.empty_cache()
        line["secondary"] = sec
    if not args.no_cpu_baseline:
        v, sample, threads = oracle_rate(args.workload)
        line["cpu_baseline"] = {"value": v, "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)
    for m_ in models.values():
        m_.close()


if __name__ == "__main__":
    main()
