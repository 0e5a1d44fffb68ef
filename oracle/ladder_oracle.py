"""CPU oracle for the Ladder Transformer forward pass (prefill and single-token decode).

TEST INFRASTRUCTURE ONLY.  This module exists to prove the CUDA path right.  Only
the test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline /
reference legs of ``bench.py`` may import it.  The library never calls it, and it
imports nothing from the library except the shared seeded-input generator
(``ladder_residual_transformer_gb300.synth``), which holds no model arithmetic.

It is plain and slow on purpose: numpy, one sequence and one head at a time,
library matmuls as the only building block, no fusion, no blocking, no
reordering.  Arithmetic runs in ``dtype`` (fp32 by default; fp64 to bound the
oracle's own rounding).  Weights are the bf16 values of the generator, widened
exactly.

Sources (pages on the Ladder Residual paper, arXiv 2501.06589):
  [notes]  "Ladder Residual: Parallelism-Aware Architecture for Accelerating Large
           Model Inference" (ICML 2025 paper notes).  Section 研究背景与动机
           ("core idea"): the standard update x_{i+1} = h_{i+1}(x_i) + x_i
           becomes x_{i+1} = h_{i+1}(x_{i-1}) + x_i.  Section 方法详解 / 整体框架:
           each attention or MLP module reads the stream from one module further
           back, while the stream itself still accumulates every module output.
           Section 关键设计: the staggered residual; the asynchronous all-reduce
           whose handle the next module waits on; the hybrid adaptation that keeps
           the lower layers unchanged and makes only the upper layers ladder.
  [record] "Ladder-residual: parallelism-aware architecture for accelerating large
           model inference with communication overlapping" (codewithpapers record):
           abstract, and the names of the official code's helpers (repeat_kv,
           precompute_freqs_cis / apply_rotary_emb, rotate_half, sample), which fix
           grouped-query attention, rotary embeddings and sampling as sub-steps.

Readings where the pages are silent (each one is a switch or a documented choice):
  R1  x_{-1} := x_0, so the first two ladder modules both read the embedding.
      The async-handle scheme of [notes] 关键设计 (pending outputs start empty)
      gives exactly this.
  R2  Hybrid boundary: with b = 2 * n_standard_layers, ladder module k reads
      x_{max(k-2, b)}; ``strict_boundary=True`` reads x_{k-2} instead.
  R3  Module internals follow the Llama-3.1 base that [notes] adapts: pre-norm
      RMSNorm (eps inside the square root), no biases, SwiGLU MLP, causal GQA
      attention with rotary embeddings.
  R4  Rotary pairs are interleaved (2j, 2j+1) (precompute_freqs_cis /
      apply_rotary_emb in [record]); ``rope_interleaved=0`` takes the half-split
      pairing of rotate_half.  Angles p * theta^(-2j/hd) are formed in fp64.
  R5  GQA: query head h reads KV head h // (n_q_heads / n_kv_heads) (repeat_kv).
  R6  Prefill returns the logits of each sequence's last position; greedy
      decoding takes argmax with the lowest index on ties.
  R8  Sampling beyond greedy: [record] names the official benchmark's
      logits_to_probs / multinomial_sample_one_no_sync / sample helpers (the
      gpt-fast generation loop).  Read plainly: scale the logits by 1/T (T
      clamped below at 1e-5), keep the logits at or above the k-th largest
      (top_k <= 0 or >= V keeps all), normalise to probabilities p, and return
      argmax_i p_i / q_i with q_i ~ Exp(1) drawn independently per vocabulary
      entry (the "exponential race", a sample of p).  In the log domain this is
      argmax_i l_i / T - ln(q_i).  The draws are not the pages': q_i = -ln u_i
      with u_i from SplitMix64 counters keyed by (seed, batch row, position of
      the sampled token), as written in ``sample_uniforms``.
  R9  Rotary frequency scaling: [record] names the official code's
      apply_rope_scaling helper (Llama-3.1 checkpoints).  Read as the published
      Llama-3.1 rule, written out in ``rope_inv_freq``: with wavelength
      w_j = 2 pi / f_j, frequencies with w_j < L / high_freq_factor stay,
      those with w_j > L / low_freq_factor are divided by `factor`, and those
      in between are interpolated, f = (1 - s) f / factor + s f with
      s = (L / w_j - low_freq_factor) / (high_freq_factor - low_freq_factor),
      L = the original maximum position.  ``dims["rope_scaling"]`` (a dict of
      factor, low_freq_factor, high_freq_factor, original_max_position)
      switches it on; absent or None leaves the frequencies unscaled.
  R7  The parallel-block model that [notes] compares against (the Parallel-70B
      row of the 70B latency breakdown table, section 实验关键数据) is not spelt
      out there; it is read as the usual parallel attention + MLP layer: both
      modules of layer l read the layer input x_{2l}, each through its own
      RMSNorm gain, and the stream still accumulates every module output
      (x_{2l+1} = x_{2l} + A, x_{2l+2} = x_{2l+1} + M).  ``parallel=True``
      applies it to every layer.

Pins that tie this code to something other than itself live in
tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable

import numpy as np

from ladder_residual_transformer_gb300 import synth

__all__ = [
    "OracleWeights", "synthetic_weights", "SeqCache", "rmsnorm", "rope_tables", "apply_rope",
    "causal_gqa_attention", "attention_module", "mlp_module", "silu", "module_input_index",
    "forward", "prefill", "decode_step", "greedy_generate", "teacher_forced_decode",
    "argmax_lowest", "kv_slot", "kv_pool_offset", "splitmix64_mix", "sample_uniforms", "sample_token",
    "rope_inv_freq",
]


# ---------------------------------------------------------------------------
# Weights
# ---------------------------------------------------------------------------
@dataclass
class LayerWeights:
    attn_norm: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    mlp_norm: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray


class OracleWeights:
    """Weights in the oracle's dtype, produced on demand by ``source(name, layer)``.

    ``source`` returns an array of the tensor's shape (any float dtype).  Layers
    are kept after first use unless ``keep_layers`` is False, in which case only
    the most recently used layer is kept and any other ``layer(l)`` call produces
    its weights again (used for models larger than host RAM).
    """

    def __init__(self, dims: dict, source: Callable[[str, int], np.ndarray],
                 dtype=np.float32, keep_layers: bool = True):
        self.dims = dict(dims)
        self.dtype = np.dtype(dtype)
        self._source = source
        self._keep = keep_layers
        self._layers: dict[int, LayerWeights] = {}
        self._global: dict[str, np.ndarray] = {}

    def _get(self, name: str, layer: int = -1) -> np.ndarray:
        return np.ascontiguousarray(self._source(name, layer), dtype=self.dtype)

    def glob(self, name: str) -> np.ndarray:
        if name == "lm_head" and self.dims.get("tie_embeddings"):
            name = "embed"
        if name not in self._global:
            self._global[name] = self._get(name)
        return self._global[name]

    def layer(self, l: int) -> LayerWeights:
        if l in self._layers:
            return self._layers[l]
        if not self._keep:
            self._layers.clear()  # drop the previous layer before producing the next one
        lw = LayerWeights(**{k: self._get(k, l) for k in synth.LAYER_KINDS})
        self._layers[l] = lw
        return lw


def synthetic_weights(dims: dict, seed: int = synth.WEIGHT_SEED, dtype=np.float32,
                      transform: Callable[[str, int, np.ndarray], np.ndarray] | None = None,
                      keep_layers: bool = True) -> OracleWeights:
    """The generator's bf16 weights widened exactly to ``dtype``.

    ``transform(name, layer, array)`` may replace a tensor (tests zero whole
    modules with it).
    """
    def source(name, layer):
        a = synth.gen_tensor_f32(dims, name, layer, seed=seed)
        if transform is not None:
            a = transform(name, layer, a)
        return a
    return OracleWeights(dims, source, dtype=dtype, keep_layers=keep_layers)


# ---------------------------------------------------------------------------
# Sub-steps (R3-R5)
# ---------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """n(x; g)_j = x_j / sqrt(mean_i x_i^2 + eps) * g_j over the last axis (R3)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + x.dtype.type(eps)) * g


def rope_inv_freq(head_dim: int, theta: float, scaling: dict | None = None) -> np.ndarray:
    """f_j = theta^(-2j/hd), j < hd/2, in fp64 (R4), then the frequency scaling of R9."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    f = float(theta) ** (-2.0 * j / head_dim)
    if not scaling:
        return f
    factor = float(scaling["factor"])
    low, high = float(scaling["low_freq_factor"]), float(scaling["high_freq_factor"])
    L = float(scaling["original_max_position"])
    out = np.empty_like(f)
    for i, fj in enumerate(f):
        w = 2.0 * math.pi / fj
        if w < L / high:
            out[i] = fj
        elif w > L / low:
            out[i] = fj / factor
        else:
            s = (L / w - low) / (high - low)
            out[i] = (1.0 - s) * fj / factor + s * fj
    return out


def rope_tables(positions: np.ndarray, head_dim: int, theta: float, dtype,
                scaling: dict | None = None) -> tuple[np.ndarray, np.ndarray]:
    """cos and sin of phi[p, j] = p * f_j, j < hd/2, formed in fp64 (R4, R9)."""
    inv_freq = rope_inv_freq(head_dim, theta, scaling)
    phi = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(phi).astype(dtype), np.sin(phi).astype(dtype)


def apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray, interleaved: bool = True) -> np.ndarray:
    """Rotate each pair (a, b) of every head to (a cos - b sin, a sin + b cos).

    x is [T, H, hd]; cos/sin are [T, hd/2].  Pairs are (2j, 2j+1) when
    interleaved, (j, j + hd/2) otherwise (R4).
    """
    hd = x.shape[-1]
    if interleaved:
        a, b = x[..., 0::2], x[..., 1::2]
    else:
        a, b = x[..., : hd // 2], x[..., hd // 2:]
    c, s = cos[:, None, :], sin[:, None, :]
    ra = a * c - b * s
    rb = a * s + b * c
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., : hd // 2], out[..., hd // 2:] = ra, rb
    return out


def causal_gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                         q_pos: np.ndarray, k_pos: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(hd)) v over keys at positions <= the query's (R3, R5).

    q is [T, nq, hd]; k and v are [S, nkv, hd]; query head h reads KV head
    h // (nq / nkv).  Softmax subtracts the row maximum before exponentiating.
    """
    T, nq, hd = q.shape
    nkv = k.shape[1]
    group = nq // nkv
    scale = q.dtype.type(1.0 / math.sqrt(hd))
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    out = np.empty_like(q)
    for h in range(nq):
        kh = h // group
        s = (q[:, h, :] @ k[:, kh, :].T) * scale
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kh, :]
    return out


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + e^{-z})."""
    with np.errstate(over="ignore"):
        return z / (z.dtype.type(1) + np.exp(-z))


@dataclass
class SeqCache:
    """Keys (after rotation) and values of one sequence, per layer, fp (oracle dtype)."""
    k: list = field(default_factory=list)   # per layer: [S, nkv, hd]
    v: list = field(default_factory=list)

    @property
    def length(self) -> int:
        return 0 if not self.k or self.k[0] is None else self.k[0].shape[0]


def attention_module(dims: dict, lw: LayerWeights, u: np.ndarray, start: int,
                     cache: SeqCache, layer: int) -> np.ndarray:
    """Attention module h(u) for the block of T tokens at positions start..start+T-1.

    Appends the block's rotated keys and its values to ``cache`` (layer ``layer``)
    and attends over everything cached so far.
    """
    T = u.shape[0]
    nq, nkv, hd = dims["n_q_heads"], dims["n_kv_heads"], dims["head_dim"]
    q = (u @ lw.wq.T).reshape(T, nq, hd)
    k = (u @ lw.wk.T).reshape(T, nkv, hd)
    v = (u @ lw.wv.T).reshape(T, nkv, hd)
    pos = np.arange(start, start + T)
    cos, sin = rope_tables(pos, hd, dims["rope_theta"], u.dtype, dims.get("rope_scaling"))
    inter = bool(dims.get("rope_interleaved", 1))
    q = apply_rope(q, cos, sin, inter)
    k = apply_rope(k, cos, sin, inter)
    while len(cache.k) <= layer:
        cache.k.append(None)
        cache.v.append(None)
    if cache.k[layer] is None:
        assert start == 0
        cache.k[layer], cache.v[layer] = k, v
    else:
        assert cache.k[layer].shape[0] == start
        cache.k[layer] = np.concatenate([cache.k[layer], k], axis=0)
        cache.v[layer] = np.concatenate([cache.v[layer], v], axis=0)
    kk, vv = cache.k[layer], cache.v[layer]
    o = causal_gqa_attention(q, kk, vv, pos, np.arange(kk.shape[0]))
    return o.reshape(T, nq * hd) @ lw.wo.T


def mlp_module(lw: LayerWeights, u: np.ndarray) -> np.ndarray:
    """SwiGLU MLP: W_down (silu(W_gate u) * (W_up u)) (R3)."""
    return (silu(u @ lw.w_gate.T) * (u @ lw.w_up.T)) @ lw.w_down.T


# ---------------------------------------------------------------------------
# The ladder schedule ([notes] 研究背景与动机, 方法详解, 关键设计; R1, R2)
# ---------------------------------------------------------------------------
def module_input_index(k: int, n_standard_layers: int, strict_boundary: bool = False,
                       parallel: bool = False) -> int:
    """Index j of the stream state x_j that module k (1-based) reads.

    Module k is the attention (k odd) or MLP (k even) of layer (k-1)//2.  In a
    standard layer it reads x_{k-1}; in a ladder layer it reads x_{k-2} (the
    staggered residual of [notes]), with x_{-1} := x_0 (R1) and the hybrid
    boundary rule R2.  With ``parallel`` every layer is a parallel block (R7):
    both modules of layer l read x_{2l}.
    """
    if parallel:
        return k - 1 if k % 2 == 1 else k - 2
    layer = (k - 1) // 2
    if layer < n_standard_layers:
        return k - 1
    if strict_boundary:
        return max(k - 2, 0)
    return max(k - 2, 2 * n_standard_layers)


def forward(dims: dict, W: OracleWeights, blocks: list[np.ndarray], caches: list[SeqCache],
            all_positions: bool = False, strict_boundary: bool = False,
            return_stream: bool = False, parallel: bool = False):
    """Run one block of new tokens per sequence through the model.

    blocks[b] holds the token ids that sequence b appends, at positions
    caches[b].length onward.  The stream x_0 = E[tok]; module k computes
    x_k = x_{k-1} + h_k(n(x_{j(k)}; g_k)) with j from ``module_input_index``.
    Returns the logits of each block's last position ([B, V]), or of every
    position (list of [T_b, V]) with ``all_positions``.
    """
    L = dims["n_layers"]
    nstd = dims["n_standard_layers"]
    eps = dims["norm_eps"]
    dt = W.dtype
    E = W.glob("embed")
    starts = [c.length for c in caches]
    # hist[b][j] = x_j of sequence b.
    hist = [[E[np.asarray(blk, dtype=np.int64)].astype(dt)] for blk in blocks]
    for k in range(1, 2 * L + 1):
        layer = (k - 1) // 2
        lw = W.layer(layer)
        j = module_input_index(k, nstd, strict_boundary, parallel)
        for b in range(len(blocks)):
            if len(blocks[b]) == 0:
                hist[b].append(hist[b][-1])
                continue
            x_in = hist[b][j]
            if k % 2 == 1:
                u = rmsnorm(x_in, lw.attn_norm, eps)
                h = attention_module(dims, lw, u, starts[b], caches[b], layer)
            else:
                u = rmsnorm(x_in, lw.mlp_norm, eps)
                h = mlp_module(lw, u)
            hist[b].append(hist[b][k - 1] + h)
    gf = W.glob("final_norm")
    Wlm = W.glob("lm_head")
    outs = []
    for b in range(len(blocks)):
        xL = hist[b][2 * L]
        if not all_positions:
            xL = xL[-1:]
        logits = rmsnorm(xL, gf, eps) @ Wlm.T
        outs.append(logits if all_positions else logits[0])
    if return_stream:
        return (outs if all_positions else np.stack(outs)), hist
    return outs if all_positions else np.stack(outs)


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Greedy token: index of the largest logit, the lowest index on ties (R6)."""
    return np.argmax(logits, axis=-1).astype(np.int32)


# ---------------------------------------------------------------------------
# Sampling (R8)
# ---------------------------------------------------------------------------
_M64 = (1 << 64) - 1
SM64_GAMMA = 0x9E3779B97F4A7C15


def splitmix64_mix(z):
    """The SplitMix64 output function (Steele, Lea and Flood, "Fast splittable
    pseudorandom number generators", OOPSLA 2014), on Python ints or uint64
    arrays (arithmetic modulo 2^64)."""
    if isinstance(z, np.ndarray):
        with np.errstate(over="ignore"):
            z = z.astype(np.uint64)
            z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
            z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
            return z ^ (z >> np.uint64(31))
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def sample_uniforms(seed: int, row: int, pos: int, n: int) -> np.ndarray:
    """u_i, i < n, for batch row `row` sampling the token at position `pos`:
    key = mix(mix(seed + G (row + 1)) + G (pos + 1)), u_i = (top 23 bits of
    mix(key + G (i + 1)) + 1/2) / 2^23, with G the SplitMix64 increment.  Every
    u_i lies in (0, 1) and is exact in fp32 and fp64."""
    k1 = splitmix64_mix((seed + SM64_GAMMA * (row + 1)) & _M64)
    key = splitmix64_mix((k1 + SM64_GAMMA * (pos + 1)) & _M64)
    with np.errstate(over="ignore"):
        ctr = np.uint64(key) + np.uint64(SM64_GAMMA) * np.arange(1, n + 1, dtype=np.uint64)
    h = splitmix64_mix(ctr)
    return ((h >> np.uint64(41)).astype(np.float64) + 0.5) / float(1 << 23)


def sample_token(logits_row: np.ndarray, temperature: float, top_k: int, seed: int, row: int, pos: int,
                 return_scores: bool = False):
    """Next token of one row by temperature / top-k sampling (R8); greedy when
    temperature <= 0.  Scores l_i / T - ln(-ln u_i) in fp64, -inf outside the
    top-k set; the lowest index wins ties."""
    l = np.asarray(logits_row, dtype=np.float64)
    V = l.shape[0]
    if temperature <= 0:
        tok = int(np.argmax(l))
        return (tok, l) if return_scores else tok
    T = max(float(temperature), 1e-5)
    keep = np.ones(V, dtype=bool)
    if 0 < top_k < V:
        pivot = np.sort(l)[V - top_k]  # the k-th largest logit
        keep = l >= pivot
    u = sample_uniforms(seed, row, pos, V)
    score = np.where(keep, l / T - np.log(-np.log(u)), -np.inf)
    tok = int(np.argmax(score))
    return (tok, score) if return_scores else tok


def prefill(dims: dict, W: OracleWeights, prompts: list[np.ndarray], **kw):
    """Prefill from empty caches; returns (last-position logits [B, V], caches)."""
    caches = [SeqCache() for _ in prompts]
    logits = forward(dims, W, prompts, caches, **kw)
    return logits, caches


def decode_step(dims: dict, W: OracleWeights, tokens: np.ndarray, caches: list[SeqCache], **kw):
    """One token per sequence at position caches[b].length; returns logits [B, V]."""
    return forward(dims, W, [np.asarray([t]) for t in tokens], caches, **kw)


def greedy_generate(dims: dict, W: OracleWeights, prompts: list[np.ndarray], steps: int, **kw):
    """Prefill, then ``steps`` decode steps each fed the previous greedy token.

    Returns (tokens [B, steps + 1], logits [steps + 1, B, V], caches).
    """
    logits, caches = prefill(dims, W, prompts, **kw)
    toks = [argmax_lowest(logits)]
    all_logits = [logits]
    for _ in range(steps):
        logits = decode_step(dims, W, toks[-1], caches, **kw)
        all_logits.append(logits)
        toks.append(argmax_lowest(logits))
    return np.stack(toks, axis=1), np.stack(all_logits), caches


def teacher_forced_decode(dims: dict, W: OracleWeights, prompts: list[np.ndarray],
                          feed: np.ndarray, **kw):
    """Prefill, then decode feeding feed[:, s] at step s; returns logits [S + 1, B, V]."""
    logits, caches = prefill(dims, W, prompts, **kw)
    out = [logits]
    for s in range(feed.shape[1]):
        out.append(decode_step(dims, W, feed[:, s], caches, **kw))
    return np.stack(out), caches


# ---------------------------------------------------------------------------
# Paged KV-cache indexing (the library's documented pool layout)
# ---------------------------------------------------------------------------
def kv_slot(block_table_row: np.ndarray, p: int, page_size: int) -> tuple[int, int]:
    """(physical page, offset in page) of position p of a sequence."""
    return int(block_table_row[p // page_size]), p % page_size


def kv_pool_offset(n_kv_heads: int, head_dim: int, num_pages: int, page_size: int,
                   layer: int, page: int, kv: int, head: int, off: int) -> int:
    """Element offset of (layer, page, K=0/V=1, head, off, 0) in the pool
    [layer][page][2][n_kv_heads][page_size][head_dim]."""
    return ((((layer * num_pages + page) * 2 + kv) * n_kv_heads + head) * page_size + off) * head_dim
