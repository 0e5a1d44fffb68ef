"""Launch timeline of one eager decode step, printed as text.

    python -m ladder_residual_transformer_gb300.timeline --workload 8b-ladder --layers 2

Builds the workload's model on synthetic weights, prefills a prompt, runs a few
decode steps, then records one eager step with the library's launch timeline
(an event pair around every projection, attention and reduce launch, on the
stream it runs on) under the configured schedule and under the standard one.
For each launch it prints the stream, the kernel class and the start and end
in microseconds after the step began, and a lane chart; in shard mode the
reduce of module k on the second stream overlaps the projections of module
k + 1 on the first when the schedule is ladder, and does not when it is
standard.  The event records between kernels defeat programmatic dependent
launch, so absolute times are longer than in a CUDA-graph step.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import ladder, synth


def record(model, tok, logits, stream, standard: bool, max_launches: int = 4096):
    with torch.cuda.stream(stream):
        model.set_mode(standard=standard, graph=False)
        for _ in range(2):
            model.decode_step(tok, logits, tok, stream)
        model.timeline_begin(max_launches, stream)
        model.decode_step(tok, logits, tok, stream)
        rows = model.timeline_end()
    stream.synchronize()
    return rows


def chart(rows, width: int = 100) -> list[str]:
    """One line per stream: a character per time bucket, the class initial of the
    launch that covers it (q qkv, a attention, o out, g gate/up, d down, r reduce,
    l lm_head), '.' when idle."""
    t_end = max(r[3] for r in rows)
    scale = width / t_end
    lines = []
    for s in (0, 1):
        lane = ["."] * width
        for st, cls, t0, t1 in rows:
            if st != s:
                continue
            for x in range(int(t0 * scale), max(int(t1 * scale), int(t0 * scale) + 1)):
                if x < width:
                    lane[x] = cls[0]
        lines.append(f"stream {s}: " + "".join(lane))
    lines.append(f"({t_end * 1e3:.0f} us across {width} columns)")
    return lines


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="8b-ladder", choices=sorted(synth.PRESETS))
    ap.add_argument("--layers", type=int, default=2, help="model depth (the workload's dims otherwise)")
    ap.add_argument("--shard-k", type=int, default=None)
    ap.add_argument("--prompt", type=int, default=2048)
    args = ap.parse_args(argv)
    dims = dict(synth.PRESETS[args.workload])
    if args.layers:
        dims["n_layers"] = args.layers
        dims["n_standard_layers"] = min(dims["n_standard_layers"], args.layers)
    shard_k = synth.RUNS.get(args.workload, {}).get("shard_k", 1) if args.shard_k is None else args.shard_k
    weights = ladder.synthetic_weights(dims, device="cuda")
    model = ladder.LadderModel(dims, weights, max_batch=1, max_seq=args.prompt + 16,
                               max_prefill_tokens=args.prompt, shard_k=shard_k)
    stream = torch.cuda.Stream()
    prompt = torch.from_numpy(synth.tokens(args.prompt, dims["vocab"]).astype(np.int32)).cuda()
    logits = torch.empty(1, dims["vocab"], device="cuda")
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    print(f"# launch timeline: {args.workload}, {dims['n_layers']} layers, shard k = {shard_k}, B = 1, "
          f"context {args.prompt}")
    for standard in (False, True):
        model.reset(stream)
        with torch.cuda.stream(stream):
            model.prefill(prompt, [args.prompt], logits, tok, stream)
        rows = record(model, tok, logits, stream, standard)
        t_first = min(r[2] for r in rows)
        rows = [(s, c, t0 - t_first, t1 - t_first) for s, c, t0, t1 in rows]
        print(f"\n## schedule: {'standard' if standard else 'configured (ladder)'}; "
              f"step {max(r[3] for r in rows) * 1e3:.1f} us\n")
        print("| # | stream | class | start us | end us |")
        print("|---|---|---|---|---|")
        for i, (s, c, t0, t1) in enumerate(rows):
            print(f"| {i} | {s} | {c} | {t0 * 1e3:.1f} | {t1 * 1e3:.1f} |")
        print("\n```")
        for line in chart(rows):
            print(line)
        print("```")


if __name__ == "__main__":
    main()
