#!/usr/bin/env python3
"""Decode and prefill throughput of the Ladder Transformer forward pass on one GB300.

Headline workload: the 70B-shape Ladder Transformer (80 ladder layers, d_model
8192, 64 query / 8 KV heads of 128, SwiGLU 28672, vocab 128256, random-init
bf16-valued weights, 141 GB resident on the GPU), batch 1.  One step =
  (a) an untimed 2048-token prefill that fills the KV cache,
  (b) 64 greedy decode steps from context 2048 (timed: `value`, decode tok/s),
  (c) a 512-token prefill from an empty cache (timed: `prefill`).
Every decode step streams all 139 GB of weights and the KV cache (far more
than the 129 MB L2), so no flush is needed between steps.

The other workloads ride along as nested entries of the same line (`configs`),
each timed the same way on its own model: the 1.2B ladder model (prompt 1024,
256 decode steps; with the standard and parallel-block schedules on the same
weights), the 8B hybrid (decode at batch 1 and 16 from context 2048; prefill
of 4 x 4096 tokens), and the 8B full ladder in shard mode (k = 8; ladder vs
standard schedule, batch 1 decode from context 2048).

Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-nested]
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
DTYPE = ("fp16 storage of the bf16-valued weights; fp16 tensor-core operands (prefill GEMM activations "
         "as fp16 hi/lo pairs); fp32 accumulation and residual stream; fp16 KV cache")
DTYPE_BF16 = ("bf16 weights; bf16 tensor-core operands (prefill GEMM activations as bf16 hi/lo pairs); fp32 "
              "accumulation and residual stream; bf16 KV cache")
L2_BYTES = 129 * 10 ** 6  # GB300 L2 cache

# What each workload's step runs.  ctx: decode starts from a prompt of this many
# tokens (prefilled untimed); prefill: the timed prefill's prompt lengths.
PLANS = {
    "70b": {"decode": [{"batch": 1, "ctx": 2048, "steps": 64}], "prefill": [512]},
    "1.2b": {"decode": [{"batch": 1, "ctx": 1024, "steps": 256}], "prefill": [1024], "schedules": True},
    "8b-hybrid": {"decode": [{"batch": 1, "ctx": 2048, "steps": 128}, {"batch": 16, "ctx": 2048, "steps": 128}],
                  "prefill": [4096] * 4},
    "8b-ladder": {"decode": [{"batch": 1, "ctx": 2048, "steps": 128}], "prefill": [], "shard_k": 8},
    "tiny": {"decode": [{"batch": 1, "ctx": 16, "steps": 8}], "prefill": [16]},
    # the 1.2B workload with bf16 storage: bf16 weights, KV cache and tensor-core operands
    "1.2b-bf16": {"preset": "1.2b", "dtype": "bf16", "decode": [{"batch": 1, "ctx": 1024, "steps": 256}],
                  "prefill": [1024]},
}
NESTED = ("1.2b", "1.2b-bf16", "8b-hybrid", "8b-ladder")


def plan_dims(name):
    """Model dimensions of a workload (its preset's)."""
    return dict(synth.PRESETS[PLANS[name].get("preset", name)])

# DRAM traffic of the dominant kernel (the decode gate/up GEMV) per launch at
# each workload's shape, from one ncu capture, valid only while the kernel's
# source file is unchanged (its sha256).
NCU_TRAFFIC = {
    "70b": {"source": "ladder_residual_transformer_gb300/csrc/gemv.cu",
            "sha256": "5737a03b36f4b77671cc4130502300c7009658742c0906908fd1f0576fa3e170",
            # mean of three captured launches: 939.63 MB read + 1.00 MB written
            "bytes_per_launch": 940626517},
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


_T0 = time.perf_counter()


def log(msg):
    """Progress on stderr (the JSON line is the only stdout output)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f} s] {msg}", file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------
def sample_dims(dims, layers):
    """The first `layers` layers of a workload (every layer has the same shapes)."""
    out = dict(dims, n_layers=min(layers, dims["n_layers"]))
    out["n_standard_layers"] = min(dims["n_standard_layers"], out["n_layers"])
    return out


def oracle_sample(dims, prompt_len, decode_steps, layers=None, W=None):
    """Time the oracle on a prefill of `prompt_len` tokens and `decode_steps`
    greedy decode steps of the workload cut to its first `layers` layers (all
    when None; weights generated before timing), and scale the measured times
    to the full depth by the ratio of algorithmic work: weight bytes per decode
    step (the oracle's decode is a chain of matrix-vector products over fp32
    weights) and flops per prefill.  Returns a dict with prefill / decode tok/s
    at full depth, the seconds timed, and the weights for reuse."""
    import oracle.ladder_oracle as O
    sd = sample_dims(dims, layers or dims["n_layers"])
    if W is None:
        W = O.synthetic_weights(sd)
        for l in range(sd["n_layers"]):
            W.layer(l)
        W.glob("embed"), W.glob("lm_head"), W.glob("final_norm")
    prompt = [synth.tokens(prompt_len, sd["vocab"])]
    t0 = time.perf_counter()
    logits, caches = O.prefill(sd, W, prompt)
    t1 = time.perf_counter()
    tok = O.argmax_lowest(logits)
    for _ in range(decode_steps):
        tok = O.argmax_lowest(O.decode_step(sd, W, tok, caches))
    t2 = time.perf_counter()
    dec_scale = (decode_step_bytes(dims, [prompt_len]) / decode_step_bytes(sd, [prompt_len]))
    pre_scale = prefill_flops(dims, [prompt_len]) / prefill_flops(sd, [prompt_len])
    return {"prefill_tok_s": prompt_len / ((t1 - t0) * pre_scale),
            "decode_tok_s": decode_steps / ((t2 - t1) * dec_scale),
            "seconds": t2 - t0, "layers": sd["n_layers"], "W": W}


def sample_text(name, dims, r, prompt_len, decode_steps, threads):
    cut = (f"its first {r['layers']} of {dims['n_layers']} layers (times scaled to full depth by the ratio of "
           f"decode weight bytes and of prefill flops), " if r["layers"] < dims["n_layers"] else "")
    return (f"{name}: the oracle (fp32 numpy) on {cut}a prefill of {prompt_len} tokens "
            f"({r['prefill_tok_s']:.3g} tok/s) + {decode_steps} greedy decode steps, {threads} BLAS thread(s), "
            f"{r['seconds']:.1f} s timed, weights generated before timing")


def cpu_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


def one_core_sample(name, prompt_len, decode_steps, layers):
    """The same oracle sample in a child process limited to one BLAS thread."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", name, str(prompt_len),
           str(decode_steps), str(layers)]
    try:
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: the GPU numbers stand on their own
        return {"error": f"{type(e).__name__}: {e}"}


# Bounded oracle samples: (prompt tokens, decode steps, layers) per workload: the
# CPU baseline of our arm (one sample of about 10-20 s), and the per-step sample of
# the reference arm (small, so that 20 timed steps stay within a few minutes).
ORACLE_SAMPLES = {"70b": (64, 24, 8), "1.2b": (128, 32, 16), "8b-hybrid": (64, 16, 8), "8b-ladder": (64, 16, 8),
                  "tiny": (16, 8, 2), "1.2b-bf16": (128, 32, 16)}
REF_SAMPLES = {"70b": (32, 8, 4), "1.2b": (64, 8, 16), "8b-hybrid": (32, 8, 4), "8b-ladder": (32, 8, 4),
               "tiny": (16, 8, 2), "1.2b-bf16": (64, 8, 16)}


def cpu_baseline(name, dims):
    prompt_len, decode_steps, layers = ORACLE_SAMPLES[name]
    r = oracle_sample(dims, prompt_len, decode_steps, layers)
    out = {"value": r["decode_tok_s"], "unit": "tok/s", "cores": cpu_threads(), "kind": "oracle",
           "sample": sample_text(name, dims, r, prompt_len, decode_steps, cpu_threads()),
           "prefill_tok_s": r["prefill_tok_s"]}
    del r["W"]
    # the tiny and 1.2B workloads' oracle on one core, alongside
    for small, key in (("tiny", "one_core_tiny"), ("1.2b", "one_core_1p2b")):
        one = one_core_sample(small, *ORACLE_SAMPLES[small])
        if "error" not in one:
            one["sample"] = sample_text(small, synth.PRESETS[small], one, ORACLE_SAMPLES[small][0],
                                        ORACLE_SAMPLES[small][1], 1)
        out[key] = one
    return out


# ---------------------------------------------------------------------------
# Reference arm: the oracle, timed as it stands on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, dims):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    prompt_len, decode_steps, layers = REF_SAMPLES[args.workload]
    W = None
    for _ in range(args.warmup):
        r = oracle_sample(dims, prompt_len, decode_steps, layers, W)
        W = r["W"]
    pre, dec, secs = [], [], []
    for _ in range(args.steps):
        r = oracle_sample(dims, prompt_len, decode_steps, layers, W)
        W = r["W"]
        pre.append(r["prefill_tok_s"])
        dec.append(r["decode_tok_s"])
        secs.append(r["seconds"])
    value = len(dec) / sum(1.0 / d for d in dec)  # decode tok/s over all timed steps
    r["seconds"] = statistics.mean(secs)
    r["prefill_tok_s"] = statistics.mean(pre)
    sample = sample_text(args.workload, dims, r, prompt_len, decode_steps, cpu_threads())
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(args.workload, dims),
        "prefill": {"value": statistics.mean(pre), "unit": "tok/s"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cpu_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def workload_config(name, dims):
    plan = PLANS[name]
    cfg = {"workload": f"{name} Ladder Transformer ({dims['n_layers']} layers, "
                       f"{dims['n_standard_layers']} standard), d_model {dims['d_model']}, "
                       f"{dims['n_q_heads']}q/{dims['n_kv_heads']}kv heads x {dims['head_dim']}, "
                       f"ffn {dims['ffn_dim']}, vocab {dims['vocab']}" +
                       (f", shard mode k = {plan['shard_k']}" if plan.get("shard_k") else "") +
                       (f", {plan['dtype']} weights, KV cache and tensor-core operands" if plan.get("dtype") else ""),
           "decode": [dict(d) for d in plan["decode"]], "prefill_tokens": list(plan["prefill"]),
           "l2": ("inputs larger than L2 (all weights streamed every step)" if decode_step_bytes(dims, [0]) > L2_BYTES
                  else "weights fit in L2 (a parity-size model, not a roofline workload)")}
    return cfg


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def measure_workload(name, dims, steps, warmup, args, peaks, dev, world, headline):
    """Build the workload's model on the device and time its step (every phase
    of PLANS[name]) `steps` times after `warmup` untimed steps."""
    import torch
    from ladder_residual_transformer_gb300 import ladder

    plan = PLANS[name]
    shard_k = plan.get("shard_k", 1) if args.shard_k is None else args.shard_k
    phases = plan["decode"]
    pre_lens = list(plan["prefill"])
    max_batch = max([d["batch"] for d in phases] + [len(pre_lens)])
    max_seq = max([d["ctx"] + d["steps"] + 1 for d in phases] + pre_lens)
    max_pre = max([d["batch"] * d["ctx"] for d in phases] + [sum(pre_lens)])
    log(f"{name}: generating weights on the device")
    weights = ladder.synthetic_weights(dims, device=dev, dtype=plan.get("dtype", "fp16"))
    model = ladder.LadderModel(dims, weights, max_batch=max_batch, max_seq=max_seq, max_prefill_tokens=max_pre,
                               shard_k=shard_k)
    log(f"{name}: model ready")
    stream = torch.cuda.Stream(device=dev)
    # every input is resident on the device before any timing
    dec_in = []
    for d in phases:
        prompts = [synth.tokens(d["ctx"], dims["vocab"], stream=b) for b in range(d["batch"])]
        dec_in.append((prompts, torch.from_numpy(np.concatenate(prompts).astype(np.int32)).to(dev)))
    pre_prompts = [synth.tokens(n, dims["vocab"], stream=b) for b, n in enumerate(pre_lens)]
    pre_dev = torch.from_numpy(np.concatenate(pre_prompts).astype(np.int32)).to(dev) if pre_lens else None
    tok = torch.zeros(max_batch, dtype=torch.int32, device=dev)
    logits = torch.empty(max_batch, dims["vocab"], dtype=torch.float32, device=dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def one_step(fast_prefill=False, decode=True, prefill=True, **mode):
        """One pass over the phases; returns (decode ms per phase, prefill ms, launches)."""
        launches, d_ev, p_ev = 0, [], None
        model.set_mode(graph=not args.eager, pdl=not args.no_pdl, fast_prefill=fast_prefill, **mode)
        for d, (prompts, pdev) in zip(phases if decode else [], dec_in):
            B = d["batch"]
            model.reset(stream)
            model.prefill(pdev, [d["ctx"]] * B, logits[:B], tok[:B], stream)  # fills the context, untimed
            e0, e1 = ev(), ev()
            e0.record(stream)
            for _ in range(d["steps"]):
                model.decode_step(tok[:B], logits[:B], tok[:B], stream)
                launches += model.last_launch_count()
            e1.record(stream)
            d_ev.append((e0, e1))
        if pre_lens and prefill:
            Bp = len(pre_lens)
            model.reset(stream)
            e0, e1 = ev(), ev()
            e0.record(stream)
            model.prefill(pre_dev, pre_lens, logits[:Bp], tok[:Bp], stream)
            launches += model.last_launch_count()
            e1.record(stream)
            p_ev = (e0, e1)
        stream.synchronize()
        return ([a.elapsed_time(b) for a, b in d_ev], p_ev[0].elapsed_time(p_ev[1]) if p_ev else None, launches)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            one_step()
            log(f"{name}: warm-up step {i + 1}/{warmup}")
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        clocks = ClockSampler(torch.cuda.current_device())
        dec_ms = [[] for _ in phases]
        pre_ms, launches = [], 0
        t0 = time.perf_counter()
        for _ in range(steps):
            d, p, n = one_step()
            for i, v in enumerate(d):
                dec_ms[i].append(v)
            if p is not None:
                pre_ms.append(p)
            launches += n
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier(world)
        clk = clocks.stop()
        log(f"{name}: {steps} timed steps in {wall:.1f} s")

        # The prefill with its activations rounded once (LADDER_FLAG_FAST_PREFILL).
        fast_ms = []
        if pre_lens:
            for i in range(warmup + min(steps, 5)):
                _, p, _ = one_step(fast_prefill=True, decode=False)
                if i >= warmup:
                    fast_ms.append(p)

        # Dominant kernel of decode: time each gate/up GEMV launch over one eager
        # pass of the first decode phase.
        d0 = phases[0]
        model.set_mode(graph=False, pdl=not args.no_pdl)
        model.reset(stream)
        model.prefill(dec_in[0][1], [d0["ctx"]] * d0["batch"], logits[:d0["batch"]], tok[:d0["batch"]], stream)
        model.probe_begin("gateup", d0["steps"] * dims["n_layers"])
        for _ in range(d0["steps"]):
            model.decode_step(tok[:d0["batch"]], logits[:d0["batch"]], tok[:d0["batch"]], stream)
        n_probe, probe_ms = model.probe_end()
        stream.synchronize()

    out = {"config": workload_config(name, dims)}
    # decode phases
    out["decode"] = []
    for d, ms in zip(phases, dec_ms):
        tot = max_over_ranks([sum(ms)], world, dev)[0]
        toks = sum_over_ranks([float(d["batch"] * d["steps"] * len(ms))], world, dev)[0]
        bytes_step = statistics.mean(decode_step_bytes(dims, [d["ctx"] + i] * d["batch"]) for i in range(d["steps"]))
        gbs = bytes_step * d["steps"] * len(ms) / (sum(ms) / 1e3) / 1e9
        out["decode"].append({"batch": d["batch"], "ctx": d["ctx"], "steps": d["steps"],
                              "tok_s": toks / (tot / 1e3), "ms_per_token": sum(ms) / (d["steps"] * len(ms)),
                              "achieved_gbs": gbs, "peak_gbs": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
                              "bytes_per_step": bytes_step})
    if pre_ms:
        pf = prefill_flops(dims, pre_lens)
        tot = max_over_ranks([sum(pre_ms)], world, dev)[0]
        toks = sum_over_ranks([float(sum(pre_lens) * len(pre_ms))], world, dev)[0]
        tf = pf * len(pre_ms) / (sum(pre_ms) / 1e3) / 1e12
        ftf = pf * len(fast_ms) / (sum(fast_ms) / 1e3) / 1e12 if fast_ms else None
        out["prefill"] = {
            "value": toks / (tot / 1e3), "unit": "tok/s", "ms": sum(pre_ms) / len(pre_ms), "tokens": pre_lens,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "flops": pf,
                         "note": "algorithmic flops (2 x rows x weights + causal attention + last-row lm_head); "
                                 "the hi/lo activation operands issue twice the GEMM tensor-core work"},
            "fast": {"ms": statistics.mean(fast_ms), "tok_s": sum(pre_lens) / (statistics.mean(fast_ms) / 1e3),
                     "achieved_tflops": ftf, "frac": ftf / peaks["bf16_tflops"],
                     "note": "LADDER_FLAG_FAST_PREFILL: activations rounded once to 16 bits"} if fast_ms else None}
    gu_bytes = 2 * 2 * dims["ffn_dim"] * dims["d_model"]  # gate + up rows, 16-bit
    gu_s = probe_ms / max(n_probe, 1) / 1e3
    gu_gbs = gu_bytes / gu_s / 1e9 if gu_s > 0 else None
    traffic = None
    t = NCU_TRAFFIC.get(name)
    if t and d0["batch"] == 1:
        src = os.path.join(ROOT, t["source"])
        if os.path.exists(src) and hashlib.sha256(open(src, "rb").read()).hexdigest() == t["sha256"]:
            traffic = t["bytes_per_launch"]
    out["roofline"] = {"bound": "hbm", "kernel": "decode gate/up GEMV (RMSNorm + SwiGLU fused)",
                       "achieved": gu_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "frac": gu_gbs / peaks["hbm_gbs"] if gu_gbs else None, "traffic": traffic,
                       "algorithmic_bytes_per_launch": gu_bytes, "launches_timed": n_probe,
                       "timing": "CUDA events on the launching stream around each launch, one eager pass of the "
                                 "first decode phase right after the timed region"}
    out["clocks"] = clk
    out["gpu_launches"] = launches
    out["wall_s"] = wall
    out["steps"], out["warmup"] = steps, warmup
    out["ms_per_step"] = (sum(sum(m) for m in dec_ms) + sum(pre_ms)) / steps

    log(f"{name}: fast prefill and gate/up probe done")
    # the same weights and kernels under the other residual schedules
    ns = min(steps, 5)
    if plan.get("schedules") and not args.no_schedules:
        sch = {}
        for label, mode in (("standard", {"standard": True}), ("parallel", {"parallel": True})):
            d_all, p_all = [], []
            for i in range(warmup + ns):
                d, p, _ = one_step(**mode)
                if i >= warmup:
                    d_all.append(d[0])
                    p_all.append(p)
            sch[label] = {"decode_tok_s": phases[0]["batch"] * phases[0]["steps"] * ns / (sum(d_all) / 1e3),
                          "prefill_ms": statistics.mean(p_all) if p_all[0] is not None else None}
        sch["configured"] = {"decode_tok_s": out["decode"][0]["tok_s"] / world,
                             "prefill_ms": out["prefill"]["ms"] if pre_ms else None}
        sch["note"] = ("same weights and kernels; configured = the workload's ladder/hybrid schedule; standard = "
                       "every layer standard; parallel = every layer a parallel attention + MLP block")
        out["schedules"] = sch
    if shard_k > 1 and not args.no_schedules:
        d_all = []
        for i in range(warmup + ns):
            d, _, _ = one_step(prefill=False, standard=True)
            if i >= warmup:
                d_all.append(d[0])
        out["shard"] = {"k": shard_k, "ladder_decode_tok_s": out["decode"][0]["tok_s"] / world,
                        "standard_decode_tok_s": phases[0]["batch"] * phases[0]["steps"] * ns / (sum(d_all) / 1e3),
                        "note": "same weights and kernels; standard = every module waits for the previous "
                                "module's reduce; ladder = each module waits for the reduce two modules back"}

    # end to end through the host API: host prompt in, host tokens out
    if headline and not args.no_e2e:
        prompts = dec_in[0][0]
        reps = min(steps, 5)
        with torch.cuda.stream(stream):
            model.set_mode(graph=not args.eager, pdl=not args.no_pdl)
            model.generate(prompts, d0["steps"], stream)
            ts = []
            for _ in range(reps):
                t = time.perf_counter()
                model.generate(prompts, d0["steps"], stream)
                ts.append(time.perf_counter() - t)
        tmax = max_over_ranks([sum(ts)], world, dev)[0]
        gen = sum_over_ranks([float(d0["batch"] * d0["steps"] * reps)], world, dev)[0]
        out["e2e"] = {"value": gen / tmax, "unit": "tok/s",
                      "timed": f"generate(): pinned H2D of the {d0['ctx']}-token prompt, its prefill, "
                               f"{d0['steps']} decode steps, D2H of the tokens; wall clock, prefill included",
                      "h2d_bytes_per_step": 4 * d0["batch"] * d0["ctx"],
                      "d2h_bytes_per_step": 4 * d0["batch"] * (d0["steps"] + 1)}
    model.close()
    del model, weights
    torch.cuda.empty_cache()
    log(f"{name}: done")
    return out


def run_ours(args, dims):
    import torch

    rank, world, local = dist_env()
    dist_init(world, "nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    peaks, peak_src = load_peaks()
    t_start = time.perf_counter()
    head = measure_workload(args.workload, dims, args.steps, args.warmup, args, peaks, dev, world, headline=True)
    nested = {}
    if not args.no_nested and args.workload == "70b":
        for name in NESTED:
            try:
                nested[name] = measure_workload(name, plan_dims(name), min(args.steps, 5),
                                                max(3, min(args.warmup, 3)), args, peaks, dev, world, headline=False)
            except Exception as e:  # recorded in the line; the headline stands
                nested[name] = {"error": f"{type(e).__name__}: {e}"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        log("oracle baseline on the host cores")
        cpu = cpu_baseline(args.workload, dims)
        log("oracle baseline done")
    d0 = head["decode"][0]
    plan = PLANS[args.workload]
    out = {
        "metric": METRIC, "value": d0["tok_s"], "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_BF16 if plan.get("dtype") == "bf16" else DTYPE,
        "data": "synthetic (random-init weights, random tokens)",
        "config": dict(head["config"], batch=plan["decode"][0]["batch"], decode_ctx=plan["decode"][0]["ctx"],
                       decode_steps=plan["decode"][0]["steps"], parallelism=f"replicas x{world}",
                       decode_launch=("eager" if args.eager else "cuda graph") + (", no PDL" if args.no_pdl else ", PDL"),
                       step=("untimed prefill of the decode context, timed decode steps, timed prefill of "
                             "prefill_tokens from an empty cache")),
        "decode": d0,
        "prefill": head.get("prefill"),
        "roofline": head["roofline"],
        "peaks": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'fallback 6.8 TB/s, 1.9 PF bf16'})",
        "gpu_launches": head["gpu_launches"], "clocks": head["clocks"], "e2e": head.get("e2e"),
        "cpu_baseline": cpu,
        "shard": head.get("shard"), "schedules": head.get("schedules"),
        "configs": nested or None,
        "wall_s": time.perf_counter() - t_start,
    }
    if len(head["decode"]) > 1:
        out["decode_phases"] = head["decode"]
    return out if rank == 0 else None


def main():
    if len(sys.argv) > 1 and sys.argv[1] == "--oracle-sample":
        # child process of one_core_sample: name prompt decode layers -> JSON
        name, prompt_len, decode_steps, layers = sys.argv[2], int(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5])
        r = oracle_sample(dict(synth.PRESETS[name]), prompt_len, decode_steps, layers)
        del r["W"]
        print(json.dumps(dict(r, cores=1, unit="tok/s", value=r["decode_tok_s"], kind="oracle")))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="70b", choices=sorted(PLANS))
    ap.add_argument("--shard-k", type=int, default=None, help="shard mode k (default: the workload's)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="decode without programmatic dependent launch")
    ap.add_argument("--eager", action="store_true", help="decode without CUDA-graph replay")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-nested", action="store_true", help="time the named workload only")
    ap.add_argument("--layers", type=int, default=None,
                    help="cut the workload to this many layers (for kernel captures; the line names the count)")
    ap.add_argument("--no-schedules", action="store_true",
                    help="skip timing the standard and parallel-block schedules on the same weights")
    args = ap.parse_args()
    dims = plan_dims(args.workload)
    if args.layers:
        # kernel captures on a shallow copy of the workload (every layer has the same shapes)
        dims = sample_dims(dims, args.layers)
        args.no_nested = True
    out = run_reference(args, dims) if args.impl == "reference" else run_ours(args, dims)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
