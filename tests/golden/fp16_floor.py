"""Writes tests/golden/fp16_floor_8b_hybrid.json: the logit error that an exactly
rounded 16-bit-activation pipeline has against the fp32 oracle on the 8B hybrid
test inputs (prompts of 256 and 96 tokens, seed 1; weights seed 0).

The oracle's arithmetic is run unchanged except that the values a 16-bit
tensor-core pipeline stores in fp16 are rounded to fp16 (round to nearest
even) where the GPU rounds them: the normalised GEMM inputs, the attention
output, the SwiGLU output, the queries and the cached keys and values.  This
is the floor any implementation with fp16 activations reaches; it calls
nothing but the oracle and the seeded generator.

Run from the repository root:  python tests/golden/fp16_floor.py   (about a
minute per pass on 16 cores; 32 GB of fp32 weights in host memory).
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle.ladder_oracle as O  # noqa: E402
from ladder_residual_transformer_gb300 import synth  # noqa: E402


def h(x):
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def rounded_prefill(dims, W, prompts):
    keep = (O.rmsnorm, O.causal_gqa_attention, O.mlp_module)
    try:
        O.rmsnorm = lambda x, g, e: h(keep[0](x, g, e))
        O.causal_gqa_attention = lambda q, k, v, qp, kp: h(keep[1](h(q), h(k), h(v), qp, kp))
        O.mlp_module = lambda lw, u: h(O.silu(u @ lw.w_gate.T) * (u @ lw.w_up.T)) @ lw.w_down.T
        out, _ = O.prefill(dims, W, prompts)
    finally:
        O.rmsnorm, O.causal_gqa_attention, O.mlp_module = keep
    return out


if __name__ == "__main__":
    dims = dict(synth.PRESETS["8b-hybrid"])
    prompts = [synth.tokens(n, dims["vocab"], stream=b) for b, n in enumerate([256, 96])]
    W = O.synthetic_weights(dims)
    ref, _ = O.prefill(dims, W, prompts)
    got = rounded_prefill(dims, W, prompts)
    rec = {"workload": "8b-hybrid, prompts 256 + 96 tokens (seed 1), weights seed 0, prefill logits",
           "max_abs": float(np.abs(got - ref).max()),
           "rel_l2": float(np.linalg.norm(got - ref) / np.linalg.norm(ref))}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fp16_floor_8b_hybrid.json")
    json.dump(rec, open(path, "w"), indent=1)
    print(rec)
