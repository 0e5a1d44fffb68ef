"""Where 16-bit rounding moves the logits: the oracle's forward pass with chosen
intermediate values rounded to fp16, against the same pass without rounding.

TEST INFRASTRUCTURE ONLY (an analysis aid; the library never imports it).  It
uses the oracle's own sub-steps and schedule, and the seeded generator, and
nothing of the CUDA path.

A GPU forward pass with 16-bit tensor-core operands rounds values at fixed
points; each rounding adds relative noise of up to 2^-11 (fp16) that the rest
of the network carries to the logits.  Rounding one point at a time, or all
points but some, shows which points dominate the logit error and what a path
that keeps some of them wider reaches.  The points:

  u_attn  normalised rows into the QKV projection
  u_mlp   normalised rows into the gate/up projection
  a       SwiGLU output (into W_down)
  o       attention output (into W_o)
  q, k, v rotated queries and keys, values (the attention operands and the cache)
  p       softmax probabilities before P V

The variants run in lock step, layer by layer, so that each layer's weights
are generated once (deep models do not fit host memory in fp32).

  python -m oracle.rounding_attribution 70b 32            # last-position logits of a 32-token prompt
  python -m oracle.rounding_attribution 8b-hybrid 256
"""
from __future__ import annotations

import json
import math
import sys
import time

import numpy as np

from ladder_residual_transformer_gb300 import synth

from . import ladder_oracle as O

POINTS = ("u_attn", "u_mlp", "a", "o", "q", "k", "v", "p")
GEMM_OPERANDS = {"u_attn", "u_mlp", "a", "o"}


def fp16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest fp16 value (ties to even), back in fp32."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


_ORACLE_ATTENTION = O.causal_gqa_attention


def attention(q, k, v, q_pos, k_pos, points):
    """The oracle's causal GQA attention with the chosen operands rounded; its
    own function unless the probabilities are rounded too."""
    if "q" in points:
        q = fp16(q)
    if "k" in points:
        k = fp16(k)
    if "v" in points:
        v = fp16(v)
    if "p" not in points:
        out = _ORACLE_ATTENTION(q, k, v, q_pos, k_pos)
        return fp16(out) if "o" in points else out
    T, nq, hd = q.shape
    group = nq // k.shape[1]
    scale = q.dtype.type(1.0 / math.sqrt(hd))
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    out = np.empty_like(q)
    for h in range(nq):
        kh = h // group
        s = np.where(visible, (q[:, h, :] @ k[:, kh, :].T) * scale, -np.inf)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        total = e.sum(axis=1, keepdims=True)
        if "p" in points:
            e = fp16(e)
        out[:, h, :] = (e @ v[:, kh, :]) / total
    return fp16(out) if "o" in points else out


def attribution(dims: dict, prompt: np.ndarray, variants: dict[str, set], return_logits: bool = False):
    """(max-abs, relative L2) of each variant's last-position logits against the
    unrounded pass (variant set()); with return_logits also the logits of every
    variant, the unrounded one under "exact"."""
    L, nstd, eps = dims["n_layers"], dims["n_standard_layers"], dims["norm_eps"]
    W = O.synthetic_weights(dims, keep_layers=False)
    names = ["exact"] + list(variants)
    pts = dict(variants, exact=set())
    E = W.glob("embed")
    hist = {n: [E[prompt.astype(np.int64)].astype(np.float32)] for n in names}
    caches = {n: O.SeqCache() for n in names}
    keep = O.causal_gqa_attention
    try:
        for l in range(L):
            lw = W.layer(l)
            for k in (2 * l + 1, 2 * l + 2):
                j = O.module_input_index(k, nstd)
                for n in names:
                    p = pts[n]
                    if k % 2 == 1:
                        u = O.rmsnorm(hist[n][j], lw.attn_norm, eps)
                        u = fp16(u) if "u_attn" in p else u
                        O.causal_gqa_attention = lambda q_, k_, v_, qp, kp, p=p: attention(q_, k_, v_, qp, kp, p)
                        h = O.attention_module(dims, lw, u, 0, caches[n], l)
                    else:
                        u = O.rmsnorm(hist[n][j], lw.mlp_norm, eps)
                        u = fp16(u) if "u_mlp" in p else u
                        a = O.silu(u @ lw.w_gate.T) * (u @ lw.w_up.T)
                        h = (fp16(a) if "a" in p else a) @ lw.w_down.T
                    hist[n].append(hist[n][k - 1] + h)
                    if len(hist[n]) > 3:  # later modules read at most two states back
                        hist[n][-4] = None
    finally:
        O.causal_gqa_attention = keep
    gf, Wlm = W.glob("final_norm"), W.glob("lm_head")
    logits = {n: (O.rmsnorm(hist[n][2 * L][-1:], gf, eps) @ Wlm.T)[0] for n in names}
    ref = logits["exact"]
    res = {n: (float(np.abs(logits[n] - ref).max()), float(np.linalg.norm(logits[n] - ref) / np.linalg.norm(ref)))
           for n in variants}
    return (res, logits) if return_logits else res


DEFAULT_VARIANTS = {
    "all": set(POINTS),
    **{pt: {pt} for pt in POINTS},
    "all but the GEMM operands": set(POINTS) - GEMM_OPERANDS,
}


if __name__ == "__main__":
    preset, T = sys.argv[1], int(sys.argv[2])
    dims = dict(synth.PRESETS[preset])
    t0 = time.time()
    res = attribution(dims, synth.tokens(T, dims["vocab"]), DEFAULT_VARIANTS)
    for n, (e, r) in res.items():
        print(f"{n:28s} max-abs {e:.3e}  rel-L2 {r:.3e}")
    print(json.dumps({"workload": preset, "prompt_tokens": T, "seconds": time.time() - t0, "results": res}))
