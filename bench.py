"""Benchmark of the Qwen3-0.6B-shaped decoder pass on GB300.

Default workload (one GPU): batch-1 decode after a 512-token random prompt,
greedy, the cache growing from 512 to 512 + K positions (K = 256 covers the
512 -> 768 range).  One timed step = one full decode step: embedding, 28 blocks,
final norm, tied LM head and the greedy sampler, with the sampled id fed back on
the device as the next step's token.

Also reported (secondary, same process): batch-64 decode over ragged synthetic
caches of 128..4096 positions (sampled, T 0.7 / top-k 50 / top-p 0.9) and
prefill of 8 x 2048 tokens.

Random-init weights (seeded, N(0, 0.02)-shaped) and random token ids: no
dataset, no checkpoint.  Inputs are larger than L2 (1.19 GB of weights per
step), so no flush is needed between steps.

--impl reference times the CPU oracle (numpy float64) on the host cores on the
same workload and metric.

Run with several GPUs through torch.distributed.run: every rank runs an
independent replica (the path has no cross-GPU exchange), the timing is the max
over ranks and value counts the tokens of all ranks.
"""
from __future__ import annotations

import argparse
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
LAYER_WEIGHT_BYTES = 2 * (S.n_heads * S.head_dim * S.hidden + 2 * S.n_kv_heads * S.head_dim * S.hidden +
                          S.hidden * S.n_heads * S.head_dim + 3 * S.intermediate * S.hidden)
NORM_BYTES = 2 * (2 * S.hidden + 2 * S.head_dim)
WEIGHT_BYTES = S.n_layers * (LAYER_WEIGHT_BYTES + NORM_BYTES) + 2 * S.hidden + 2 * S.vocab * S.hidden
KV_BYTES_PER_POS = S.n_layers * 2 * S.n_kv_heads * S.head_dim * 2          # 114,688 B per cached position
LINEAR_FLOP_PER_TOKEN = 2 * S.n_layers * LAYER_WEIGHT_BYTES // 2            # 2 * weights per layer stack
PROMPT, PREFILL_B, PREFILL_T, BS64 = 512, 8, 2048, 64


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
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (getattr(self, "out", "") or "").splitlines():
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


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ our path
def bs1_decode(bd, model, K, W, world):
    """configs[1]: prompt of 512 random ids, then greedy decode steps."""
    n_pages = math.ceil((PROMPT + max(K, W) + 1) / PAGE) + 1
    kv = bd.KVPool(model, n_pages)
    bt = torch.arange(n_pages, dtype=torch.int32, device="cuda").view(1, -1)
    ids = synth.token_ids(0, 1, PROMPT, S.vocab, device="cuda")
    model.prefill(ids, torch.arange(PROMPT, dtype=torch.int32, device="cuda"), [0, PROMPT], kv, bt, None)
    params = bd.sample_params([(0.0, 1, 1.0, 0)])
    n = max(K, W)
    toks = torch.empty(n + 1, dtype=torch.int32, device="cuda")
    pos = torch.arange(PROMPT, PROMPT + n, dtype=torch.int32, device="cuda")
    model.sample(params, 0, toks[0:1])
    model.check()

    def step(i):
        model.decode_step(toks[i:i + 1], pos[i:i + 1], kv, bt, None)
        model.sample(params, i + 1, toks[i + 1:i + 2])

    for i in range(W):                       # warm-up (positions 512 .. 512+W-1, rewritten below)
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    launches0 = bd.kernel_launches()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for i in range(K):
        step(i)
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    launches = bd.kernel_launches() - launches0
    model.check()
    # per-step decode time alone (the forward kernels without the sampler), for the roofline
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record()
    for i in range(K):
        model.decode_step(toks[i:i + 1], pos[i:i + 1], kv, bt, None)
    d1.record()
    torch.cuda.synchronize()
    decode_ms = d0.elapsed_time(d1) / K
    # end to end through the public API with host buffers: pinned token/position in,
    # sampled id out, every step
    h_tok = torch.empty(1, dtype=torch.int32).pin_memory()
    h_pos = torch.empty(1, dtype=torch.int32).pin_memory()
    h_out = torch.empty(1, dtype=torch.int32).pin_memory()
    d_tok = torch.empty(1, dtype=torch.int32, device="cuda")
    d_pos = torch.empty(1, dtype=torch.int32, device="cuda")
    d_out = torch.empty(1, dtype=torch.int32, device="cuda")
    h_tok[0] = int(toks[0])
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        h_pos[0] = PROMPT + i
        d_tok.copy_(h_tok, non_blocking=True)
        d_pos.copy_(h_pos, non_blocking=True)
        model.decode_step(d_tok, d_pos, kv, bt, None)
        model.sample(params, i + 1, d_out)
        h_out.copy_(d_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        h_tok[0] = int(h_out[0])
    e2e_s = time.perf_counter() - t0
    kv_bytes = sum((PROMPT + i + 1) * KV_BYTES_PER_POS for i in range(K)) / K
    kv.close()
    return {"ms": ms, "decode_ms": decode_ms, "launches": launches, "e2e_s": e2e_s,
            "bytes_per_step": WEIGHT_BYTES + kv_bytes}


def bs64_decode(bd, model, reps=5):
    """configs[3]: 64 sequences, ragged synthetic caches of 128..4096 positions, one sampled step."""
    lens = synth.uniform_ints(0, synth.STREAM_LENGTHS, BS64, 128, 4096).tolist()
    per = 4096 // PAGE + 2
    kv = bd.KVPool(model, BS64 * per)
    pool = kv.view()
    bt = torch.arange(BS64 * per, dtype=torch.int32, device="cuda").view(BS64, per)
    for s, L in enumerate(lens):
        n_p = math.ceil(L / PAGE)
        for layer in range(S.n_layers):
            for which, std in ((0, 1.0), (1, 0.64)):
                vals = synth.kv_values(0, layer, which, s * (1 << 15) * 1024, L * 1024, std, "cuda")
                vals = torch.cat([vals.view(L, 8, 128), torch.zeros(n_p * PAGE - L, 8, 128, dtype=torch.bfloat16,
                                                                     device="cuda")])
                pool[layer, s * per:s * per + n_p, which] = vals.view(n_p, PAGE, 8, 128).permute(0, 2, 1, 3)
    toks = synth.token_ids(0, 3, BS64, S.vocab, device="cuda")
    pos = torch.tensor(lens, dtype=torch.int32, device="cuda")
    params = bd.sample_params([(0.7, 50, 0.9, s) for s in range(BS64)])
    out = torch.empty(BS64, dtype=torch.int32, device="cuda")
    for _ in range(2):
        model.decode_step(toks, pos, kv, bt, None)
        model.sample(params, 0, out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for r in range(reps):
        model.decode_step(toks, pos, kv, bt, None)
        model.sample(params, r, out)
    e1.record()
    torch.cuda.synchronize()
    model.check()
    ms = e0.elapsed_time(e1) / reps
    kv_bytes = sum((L + 1) * KV_BYTES_PER_POS for L in lens)
    kv.close()
    return {"ms": ms, "tok_s": BS64 / (ms / 1e3), "bytes": WEIGHT_BYTES + kv_bytes}


def prefill(bd, model, reps=3):
    """configs[2]: prefill only, 8 x 2048 random prompts."""
    B, T = PREFILL_B, PREFILL_T
    kv = bd.KVPool(model, B * T // PAGE)
    bt = torch.arange(B * T // PAGE, dtype=torch.int32, device="cuda").view(B, -1)
    ids = synth.token_ids(0, 2, B * T, S.vocab, device="cuda")
    pos = torch.arange(T, dtype=torch.int32, device="cuda").repeat(B)
    cu = [T * s for s in range(B + 1)]
    last = torch.empty(B, S.vocab, device="cuda")
    model.prefill(ids, pos, cu, kv, bt, last)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        model.prefill(ids, pos, cu, kv, bt, last)
    e1.record()
    torch.cuda.synchronize()
    model.check()
    ms = e0.elapsed_time(e1) / reps
    linear = LINEAR_FLOP_PER_TOKEN * B * T
    attn = 2 * S.n_heads * S.head_dim * T * T * S.n_layers * B
    kv.close()
    return {"ms": ms, "tok_s": B * T / (ms / 1e3), "linear_flop": linear, "flop": linear + attn}


# ------------------------------------------------------------------ CPU oracle
def oracle_decode_rate(max_seconds=20.0, min_steps=2):
    """Oracle decode steps per second at batch 1 after the 512-token prompt (prefill not timed)."""
    import numpy as np
    from oracle import qwen3_ref as R
    w = synth.make_weights(S)
    orc = R.Qwen3Oracle(w, S)
    ids = synth.token_ids(0, 1, PROMPT, S.vocab).numpy()
    cache = orc.new_cache()
    logits = orc.forward(ids, np.arange(PROMPT), cache, last_only=True)
    tok = int(np.argmax(logits[0]))
    t0 = time.perf_counter()
    n = 0
    while n < min_steps or time.perf_counter() - t0 < max_seconds:
        logits = orc.forward([tok], [PROMPT + n], cache, last_only=True)
        tok = int(np.argmax(logits[0]))
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n / dt, "steps": n, "seconds": dt}


def run_reference(args, world, rank):
    if rank != 0:
        return
    r = oracle_decode_rate(max_seconds=max(5.0, 2.0 * args.steps / 64))
    cores = os.cpu_count()
    line = {"metric": "decode tok/s @bs1 (Qwen3-0.6B shape, 512-token prompt, greedy)", "value": r["value"],
            "unit": "tok/s", "n_gpus": args.gpus, "steps": r["steps"], "warmup": 0,
            "ms_per_step": 1e3 / r["value"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded random-init weights and token ids)", "impl": "reference",
            "config": {"workload": "decode bs1, prompt 512, cache 512->768, greedy", "global_batch": 1,
                       "seq_len": PROMPT},
            "cpu_baseline": {"value": r["value"], "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": f"{r['steps']} decode steps after the 512-token prompt ({r['seconds']:.1f} s)"},
            "e2e": {"value": r["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true", help="skip the batch-64 decode and prefill numbers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    torch.cuda.set_device(local)
    from transformer_decode_qwen3_gb300 import binding as bd
    bd.load()
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    w = synth.make_weights(S, device="cuda")             # bit-identical to the CPU generator
    model = bd.Model(w, S, max_batch=64, max_tokens=PREFILL_B * PREFILL_T)
    del w
    torch.cuda.empty_cache()
    with ClockSampler(torch.cuda.current_device()) as clk:
        r = bs1_decode(bd, model, args.steps, args.warmup, world)
    ms_max = max_over_ranks(world, r["ms"])
    value = world * args.steps / (ms_max / 1e3)
    achieved = r["bytes_per_step"] / (r["decode_ms"] / 1e3) / 1e9
    line = {
        "metric": "decode tok/s @bs1 (Qwen3-0.6B shape, 512-token prompt, greedy)",
        "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded random-init bf16 weights and token ids)",
        "config": {"workload": "decode bs1, prompt 512, cache 512->768, greedy (configs[1])", "global_batch": world,
                   "seq_len": PROMPT, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (1.19 GB of weights streamed per step)"},
        "roofline": {"bound": "hbm", "kernel": "decode step (all forward kernels)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                     "bytes_per_step": r["bytes_per_step"]},
        "e2e": {"value": world * args.steps / r["e2e_s"], "unit": "tok/s", "h2d_bytes_per_step": 8,
                "d2h_bytes_per_step": 4},
        "gpu_launches": r["launches"],
        "clocks": clk.summary(),
    }
    if not args.no_secondary and rank == 0:
        b64 = bs64_decode(bd, model)
        pf = prefill(bd, model)
        line["secondary"] = {
            "decode_bs64": {"tok_s": b64["tok_s"], "ms_per_step": b64["ms"], "workload": "configs[3]",
                            "hbm_frac": b64["bytes"] / (b64["ms"] / 1e3) / 1e9 / hbm},
            "prefill_8x2048": {"tok_s": pf["tok_s"], "ms": pf["ms"], "workload": "configs[2]",
                               "tflops": pf["flop"] / (pf["ms"] / 1e3) / 1e12,
                               "tensor_frac_linear_of_burst": pf["linear_flop"] / (pf["ms"] / 1e3) / 1e12 / tf_burst},
        }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = oracle_decode_rate(max_seconds=15.0)
        line["cpu_baseline"] = {"value": cb["value"], "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{cb['steps']} batch-1 decode steps after the 512-token prompt "
                                          f"({cb['seconds']:.1f} s; prefill untimed)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    model.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
