#!/usr/bin/env python3
"""Decode and prefill throughput of the Ladder Transformer forward pass on one GB300.

Default workload: the 1.2B Ladder Transformer (16 ladder layers, d_model 2048,
32 query / 8 KV heads of 64, SwiGLU 8192, vocab 128256, tied embeddings,
random-init bf16 weights), batch 1, a 1024-token random prompt and 256 greedy
decode steps.  One step = one prefill of the prompt plus the 256 decode steps,
with the greedy token fed back on the device.  Every step streams the 2.47 GB
of weights (more than the 129 MB L2), so no L2 flush is needed between steps.

Prints one JSON line.  `value` is decode tokens/s over all ranks; prefill
tokens/s, the roofline of the dominant kernel, the end-to-end figure through
the host API and the CPU oracle baseline ride along.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ladder_residual_transformer_gb300 import synth  # noqa: E402

METRIC = "decode tok/s & % HBM roofline; prefill tok/s & % BF16 tensor peak (1 GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of the dominant kernel from one ncu capture, valid only while the
# kernel source is unchanged (sha256 of the file that defines it).
L2_BYTES = 129 * 10 ** 6  # GB300 L2 cache
NCU_TRAFFIC = {  # mean of the two captured launches
    "source": "ladder_residual_transformer_gb300/csrc/decode_kernels.cu",
    "sha256": "9b1e41e127b124917a06d8b238fa1c5057abf915ac462157c3231eff74ea9e39",
    "bytes_per_launch": 67253120,
}


# ---------------------------------------------------------------------------
# Algorithmic work
# ---------------------------------------------------------------------------
def layer_params(d):
    hd, nq, nkv = d["head_dim"], d["n_q_heads"], d["n_kv_heads"]
    return d["d_model"] * (nq + 2 * nkv) * hd + nq * hd * d["d_model"] + 3 * d["d_model"] * d["ffn_dim"]


def decode_step_bytes(d, ctx_per_seq):
    """Bytes one decode step must move: every layer matrix and the lm_head once,
    plus the K and V of every cached position (including the new one)."""
    w = 2 * (d["n_layers"] * layer_params(d) + d["vocab"] * d["d_model"])
    kv = sum(c + 1 for c in ctx_per_seq) * 2 * d["n_kv_heads"] * d["head_dim"] * 2 * d["n_layers"]
    return w + kv


def prefill_flops(d, lens):
    """2 M (layer weights) + causal attention (QK^T and PV) + last-row lm_head."""
    M = sum(lens)
    f = 2 * M * d["n_layers"] * layer_params(d)
    f += sum(4 * d["n_q_heads"] * d["head_dim"] * (t * (t + 1) // 2) for t in lens) * d["n_layers"]
    f += 2 * len(lens) * d["d_model"] * d["vocab"]
    return f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            raw = json.load(open(path))
            flat = {}

            def walk(o):
                if isinstance(o, dict):
                    for k, v in o.items():
                        if isinstance(v, (int, float)):
                            flat.setdefault(k, float(v))
                        else:
                            walk(v)
            walk(raw)
            if "hbm_gbs" in flat and "bf16_tflops" in flat:
                flat.setdefault("bf16_tflops_sustained", flat["bf16_tflops"])
                return flat, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Multi-rank plumbing (replicas: no collective on the data path)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(values, world, device="cpu"):
    """Element-wise max of a list of floats across ranks."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def sum_over_ranks(values, world, device="cpu"):
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t.tolist()


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------
def oracle_sample(dims, prompt_len, decode_steps, W=None):
    """Time the oracle on prefill of `prompt_len` tokens + `decode_steps` decode
    steps of the same model; returns (prefill tok/s, decode tok/s, seconds)."""
    import oracle.ladder_oracle as O
    if W is None:
        W = O.synthetic_weights(dims)
        for l in range(dims["n_layers"]):
            W.layer(l)
        W.glob("embed"), W.glob("lm_head"), W.glob("final_norm")
    prompt = [synth.tokens(prompt_len, dims["vocab"])]
    t0 = time.perf_counter()
    logits, caches = O.prefill(dims, W, prompt)
    t1 = time.perf_counter()
    tok = O.argmax_lowest(logits)
    for _ in range(decode_steps):
        tok = O.argmax_lowest(O.decode_step(dims, W, tok, caches))
    t2 = time.perf_counter()
    return prompt_len / (t1 - t0), decode_steps / (t2 - t1), t2 - t0, W


def cpu_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


# ---------------------------------------------------------------------------
# Arms
# ---------------------------------------------------------------------------
def run_reference(args, dims):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    W = None
    for _ in range(args.warmup):
        _, _, _, W = oracle_sample(dims, args.ref_prompt, args.ref_decode, W)
    pre, dec, secs = [], [], []
    for _ in range(args.steps):
        p, d, s, W = oracle_sample(dims, args.ref_prompt, args.ref_decode, W)
        pre.append(p)
        dec.append(d)
        secs.append(s)
    value = args.ref_decode * args.steps / sum(args.ref_decode / d for d in dec)
    sample = (f"{args.workload}: oracle prefill of {args.ref_prompt} tokens + {args.ref_decode} greedy decode "
              f"steps per step (fp32 numpy, weights generated before timing)")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(args, dims),
        "prefill": {"value": statistics.mean(pre), "unit": "tok/s"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cpu_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def workload_config(args, dims):
    return {"workload": f"{args.workload} Ladder Transformer ({dims['n_layers']} layers, "
                        f"{dims['n_standard_layers']} standard), d_model {dims['d_model']}, "
                        f"{dims['n_q_heads']}q/{dims['n_kv_heads']}kv heads x {dims['head_dim']}, "
                        f"ffn {dims['ffn_dim']}, vocab {dims['vocab']}",
            "batch": args.batch, "prompt_tokens": args.prompt, "decode_steps": args.decode,
            "l2": ("inputs larger than L2 (all weights streamed every step)" if decode_step_bytes(dims, [0]) > L2_BYTES
                   else "weights fit in L2 (a parity-size model, not a roofline workload)")}


def run_ours(args, dims):
    import torch
    from ladder_residual_transformer_gb300 import ladder

    rank, world, local = dist_env()
    dist_init(world, "nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    peaks, peak_src = load_peaks()

    weights = ladder.synthetic_weights(dims, device=dev)
    B = args.batch
    lens = [args.prompt] * B
    shard_k = synth.RUNS[args.workload].get("shard_k", 1) if args.shard_k is None else args.shard_k
    model = ladder.LadderModel(dims, weights, max_batch=B, max_seq=args.prompt + args.decode + 1,
                               max_prefill_tokens=sum(lens), shard_k=shard_k)
    prompts = [synth.tokens(n, dims["vocab"], stream=b) for b, n in enumerate(lens)]
    prompt_dev = torch.from_numpy(np.concatenate(prompts).astype(np.int32)).to(dev)
    stream = torch.cuda.Stream(device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    logits = torch.empty(B, dims["vocab"], dtype=torch.float32, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step(record=True):
        model.reset(stream)
        if record:
            ev[0].record(stream)
        model.prefill(prompt_dev, lens, logits, tok, stream)
        n_pre = model.last_launch_count()
        if record:
            ev[1].record(stream)
        n_dec = 0
        for _ in range(args.decode):
            model.decode_step(tok, logits, tok, stream)
            n_dec += model.last_launch_count()
        if record:
            ev[2].record(stream)
        return n_pre + n_dec

    with torch.cuda.stream(stream):
        model.set_mode(graph=not args.eager, pdl=not args.no_pdl)
        for _ in range(args.warmup):
            step(record=False)
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        clocks = ClockSampler(local)
        pre_ms, dec_ms, launches = [], [], 0
        t0 = time.perf_counter()
        for _ in range(args.steps):
            launches += step()
            stream.synchronize()
            pre_ms.append(ev[0].elapsed_time(ev[1]))
            dec_ms.append(ev[1].elapsed_time(ev[2]))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier(world)
        clk = clocks.stop()

        # Dominant kernel: time each gate/up GEMV launch over one eager step's decode.
        model.set_mode(graph=False, pdl=not args.no_pdl)
        model.reset(stream)
        model.prefill(prompt_dev, lens, logits, tok, stream)
        model.probe_begin("gateup", args.decode * dims["n_layers"])
        for _ in range(args.decode):
            model.decode_step(tok, logits, tok, stream)
        n_probe, probe_ms = model.probe_end()
        stream.synchronize()

    # The same weights and kernels under the other residual schedules (the pages'
    # comparison: standard, where every module waits for the previous one, and
    # the parallel-block model), each timed like the configured schedule above.
    def time_schedule(**mode):
        d_ms, p_ms = [], []
        with torch.cuda.stream(stream):
            model.set_mode(graph=not args.eager, pdl=not args.no_pdl, **mode)
            for i in range(args.warmup + args.steps):
                step(record=True)
                stream.synchronize()
                if i >= args.warmup:
                    p_ms.append(ev[0].elapsed_time(ev[1]))
                    d_ms.append(ev[1].elapsed_time(ev[2]))
            model.set_mode(graph=not args.eager, pdl=not args.no_pdl)
        return {"decode_tok_s": B * args.decode * len(d_ms) / (sum(d_ms) / 1e3),
                "prefill_ms": sum(p_ms) / len(p_ms)}

    schedules = None
    shard = None
    if not args.no_schedules:
        schedules = {"configured": {"decode_tok_s": B * args.decode * args.steps / (sum(dec_ms) / 1e3),
                                    "prefill_ms": sum(pre_ms) / len(pre_ms)},
                     "standard": time_schedule(standard=True),
                     "parallel": time_schedule(parallel=True),
                     "note": "same weights and kernels; configured = the workload's ladder/hybrid schedule; "
                             "standard = every layer standard; parallel = every layer a parallel "
                             "attention + MLP block"}
        if shard_k > 1:
            shard = {"k": shard_k, "ladder_decode_tok_s": schedules["configured"]["decode_tok_s"],
                     "standard_decode_tok_s": schedules["standard"]["decode_tok_s"],
                     "note": "same weights and kernels; standard = every module waits for the previous "
                             "module's reduce"}

    tot_pre, tot_dec = sum(pre_ms), sum(dec_ms)
    tot_pre, tot_dec = max_over_ranks([tot_pre, tot_dec], world, dev)
    dec_tokens = sum_over_ranks([float(B * args.decode * args.steps)], world, dev)[0]
    pre_tokens = sum_over_ranks([float(sum(lens) * args.steps)], world, dev)[0]
    decode_tps = dec_tokens / (tot_dec / 1e3)
    prefill_tps = pre_tokens / (tot_pre / 1e3)
    ms_per_step = (tot_pre + tot_dec) / args.steps

    # whole-decode and prefill rooflines
    ctx0 = args.prompt
    dec_bytes = sum(decode_step_bytes(dims, [ctx0 + i] * B) for i in range(args.decode))
    dec_gbs = dec_bytes * args.steps / (sum(dec_ms) / 1e3) / 1e9
    pf = prefill_flops(dims, lens)
    pre_tf = pf * args.steps / (sum(pre_ms) / 1e3) / 1e12

    gu_bytes = 2 * 2 * dims["ffn_dim"] * dims["d_model"]  # gate + up rows, bf16
    gu_avg_s = probe_ms / max(n_probe, 1) / 1e3
    gu_gbs = gu_bytes / gu_avg_s / 1e9 if gu_avg_s > 0 else None
    traffic = None
    if NCU_TRAFFIC and args.workload == "1.2b" and B == 1:
        src = os.path.join(ROOT, NCU_TRAFFIC["source"])
        if os.path.exists(src) and hashlib.sha256(open(src, "rb").read()).hexdigest() == NCU_TRAFFIC["sha256"]:
            traffic = NCU_TRAFFIC["bytes_per_launch"]

    # end to end through the host API: host prompt in, host tokens out
    e2e = None
    if not args.no_e2e:
        with torch.cuda.stream(stream):
            model.set_mode(graph=not args.eager, pdl=not args.no_pdl)
            model.generate(prompts, args.decode, stream)
            ts = []
            for _ in range(args.steps):
                t = time.perf_counter()
                model.generate(prompts, args.decode, stream)
                ts.append(time.perf_counter() - t)
        tmax = max_over_ranks([sum(ts)], world, dev)[0]
        e2e = {"value": dec_tokens / tmax, "unit": "tok/s",
               "timed": "generate(): pinned H2D of the prompt, prefill, decode steps, D2H of the tokens; "
                        "wall clock per step, prefill included",
               "h2d_bytes_per_step": 4 * sum(lens), "d2h_bytes_per_step": 4 * B * (args.decode + 1)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        p_tps, d_tps, secs, _ = oracle_sample(dims, args.cpu_prompt, args.cpu_decode)
        cpu = {"value": d_tps, "unit": "tok/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{args.workload}: oracle prefill of {args.cpu_prompt} tokens "
                         f"({p_tps:.1f} tok/s) + {args.cpu_decode} decode steps, fp32 numpy, "
                         f"{secs:.1f} s timed",
               "prefill_tok_s": p_tps}

    out = {
        "metric": METRIC, "value": decode_tps, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights, random tokens)",
        "config": dict(workload_config(args, dims), parallelism=f"replicas x{world}",
                       decode_launch=("eager" if args.eager else "cuda graph") + (", no PDL" if args.no_pdl else ", PDL")),
        "decode": {"tok_s": decode_tps, "achieved_gbs": dec_gbs, "peak_gbs": peaks["hbm_gbs"],
                   "frac": dec_gbs / peaks["hbm_gbs"], "bytes_per_step": dec_bytes / args.decode},
        "prefill": {"value": prefill_tps, "unit": "tok/s", "ms": tot_pre / args.steps,
                    "roofline": {"bound": "tensor", "achieved": pre_tf, "peak": peaks["bf16_tflops"],
                                 "unit": "TFLOP/s", "frac": pre_tf / peaks["bf16_tflops"], "flops": pf}},
        "roofline": {"bound": "hbm", "kernel": "decode gate/up GEMV (RMSNorm + SwiGLU fused)",
                     "achieved": gu_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gu_gbs / peaks["hbm_gbs"] if gu_gbs else None, "traffic": traffic,
                     "algorithmic_bytes_per_launch": gu_bytes, "launches_timed": n_probe,
                     "timing": "CUDA events on the launching stream around each launch, one eager "
                               "step's decode right after the timed region"},
        "peaks": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'fallback 6.8 TB/s, 1.9 PF bf16'})",
        "gpu_launches": launches, "clocks": clk, "e2e": e2e, "cpu_baseline": cpu, "shard": shard,
        "schedules": schedules,
        "wall_s": wall,
    }
    if rank == 0:
        return out
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="1.2b", choices=sorted(synth.PRESETS))
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--shard-k", type=int, default=None, help="shard mode k (default: the workload's)")
    ap.add_argument("--prompt", type=int, default=None)
    ap.add_argument("--decode", type=int, default=None)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="decode without programmatic dependent launch")
    ap.add_argument("--eager", action="store_true", help="decode without CUDA-graph replay")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="cut the workload to this many layers (for kernel captures; the line names the count)")
    ap.add_argument("--no-schedules", action="store_true",
                    help="skip timing the standard and parallel-block schedules on the same weights")
    ap.add_argument("--cpu-prompt", type=int, default=None, help="oracle sample prompt (default: the workload's)")
    ap.add_argument("--cpu-decode", type=int, default=None, help="oracle sample decode steps (default: the workload's)")
    ap.add_argument("--ref-prompt", type=int, default=64)
    ap.add_argument("--ref-decode", type=int, default=4)
    args = ap.parse_args()
    dims = dict(synth.PRESETS[args.workload])
    if args.layers:
        # kernel captures on a shallow copy of the workload (every layer has the same shapes)
        dims["n_layers"] = args.layers
        dims["n_standard_layers"] = min(dims["n_standard_layers"], args.layers // 2)
    run = synth.RUNS[args.workload]
    if args.prompt is None:
        args.prompt = run["prompt"]
    if args.decode is None:
        args.decode = run["decode_steps"]
    if args.cpu_prompt is None:
        args.cpu_prompt = args.prompt
    if args.cpu_decode is None:
        args.cpu_decode = args.decode
    out = run_reference(args, dims) if args.impl == "reference" else run_ours(args, dims)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
