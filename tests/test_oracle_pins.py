"""Pins for the CPU oracle: each test ties it to something other than itself.

The independent side is either a closed form, brute force on tiny inputs, or a
textbook Llama-style block assembled from PyTorch CPU library routines
(rms_norm, complex-number rotation, scaled_dot_product_attention, silu), all in
fp64.  Together they are chosen so that a dropped term, a wrong sign or index,
or a transposed operand anywhere in the oracle fails at least one of them.

Ladder recurrence: "Ladder Residual: Parallelism-Aware Architecture for
Accelerating Large Model Inference" (ICML 2025 paper notes), sections
研究背景与动机 (core idea) and 方法详解 / 关键设计.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import synth

TINY = synth.PRESETS["tiny"]


def small_dims(**over):
    d = dict(n_layers=2, n_standard_layers=0, d_model=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
             ffn_dim=96, vocab=97, rope_theta=10000.0, norm_eps=1e-5, rope_interleaved=1,
             tie_embeddings=0)
    d.update(over)
    return d


def random_weights(dims, seed=0, std=0.2):
    """fp64 weights with larger spread than the model init, so every module matters."""
    rng = np.random.default_rng(seed)

    def source(name, layer):
        shape = synth.tensor_shape(dims, name)
        if name in synth.NORM_KINDS:
            return 1.0 + 0.3 * rng.standard_normal(shape)
        return std * rng.standard_normal(shape)
    return O.OracleWeights(dims, source, dtype=np.float64)


# ---------------------------------------------------------------------------
# An independent textbook block built from torch library routines (fp64).
# ---------------------------------------------------------------------------
def t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def ref_norm(x, g, eps):
    return F.rms_norm(x, (x.shape[-1],), weight=g, eps=eps)


def ref_rope(x, start, theta, interleaved=True):
    # x [T, H, hd]; rotate as complex numbers z * e^{i p theta_j}
    T, H, hd = x.shape
    freqs = theta ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    pos = torch.arange(start, start + T, dtype=torch.float64)
    rot = torch.polar(torch.ones(T, hd // 2, dtype=torch.float64), torch.outer(pos, freqs))
    if interleaved:
        z = torch.view_as_complex(x.reshape(T, H, hd // 2, 2).contiguous())
        return torch.view_as_real(z * rot[:, None, :]).reshape(T, H, hd)
    z = torch.complex(x[..., : hd // 2], x[..., hd // 2:])
    z = z * rot[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def ref_attention_module(dims, lw, x_in, tokens_len):
    """Full-recompute causal attention over the whole sequence (no cache)."""
    d, nq, nkv, hd = dims["d_model"], dims["n_q_heads"], dims["n_kv_heads"], dims["head_dim"]
    u = ref_norm(x_in, t(lw.attn_norm), dims["norm_eps"])
    T = u.shape[0]
    q = F.linear(u, t(lw.wq)).reshape(T, nq, hd)
    k = F.linear(u, t(lw.wk)).reshape(T, nkv, hd)
    v = F.linear(u, t(lw.wv)).reshape(T, nkv, hd)
    inter = bool(dims["rope_interleaved"])
    q = ref_rope(q, 0, dims["rope_theta"], inter)
    k = ref_rope(k, 0, dims["rope_theta"], inter)
    o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                       v.transpose(0, 1)[None], is_causal=True, enable_gqa=True)
    o = o[0].transpose(0, 1).reshape(T, nq * hd)
    return F.linear(o, t(lw.wo))


def ref_mlp_module(dims, lw, x_in):
    u = ref_norm(x_in, t(lw.mlp_norm), dims["norm_eps"])
    return F.linear(F.silu(F.linear(u, t(lw.w_gate))) * F.linear(u, t(lw.w_up)), t(lw.w_down))


def ref_standard_forward(dims, W, tokens):
    """Textbook pre-norm decoder: x <- x + Attn(n(x)); x <- x + MLP(n(x))."""
    x = t(W.glob("embed"))[torch.as_tensor(tokens, dtype=torch.long)]
    for l in range(dims["n_layers"]):
        lw = W.layer(l)
        x = x + ref_attention_module(dims, lw, x, len(tokens))
        x = x + ref_mlp_module(dims, lw, x)
    return F.linear(ref_norm(x, t(W.glob("final_norm")), dims["norm_eps"]), t(W.glob("lm_head")))


def close(a, b, tol=1e-9):
    a, b = np.asarray(a), np.asarray(b)
    err = np.abs(a - b).max()
    assert err <= tol * max(1.0, np.abs(b).max()), err


# ---------------------------------------------------------------------------
# Pin (1): ladder on zero layers is the standard transformer.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("interleaved", [1, 0])
def test_zero_ladder_layers_is_standard_transformer(interleaved):
    dims = small_dims(n_layers=3, n_standard_layers=3, rope_interleaved=interleaved)
    W = random_weights(dims, 1)
    toks = np.array([3, 17, 5, 96, 0, 41, 41, 8, 2])
    got = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True)[0]
    want = ref_standard_forward(dims, W, toks).numpy()
    close(got, want)


def test_standard_reference_catches_a_dropped_residual():
    """Sanity of the pin itself: removing the MLP residual breaks agreement."""
    dims = small_dims(n_layers=2, n_standard_layers=2)
    W = random_weights(dims, 2)
    toks = np.array([1, 2, 3, 4])
    got = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True)[0]

    def broken(dims, W, tokens):
        x = t(W.glob("embed"))[torch.as_tensor(tokens, dtype=torch.long)]
        for l in range(dims["n_layers"]):
            lw = W.layer(l)
            x = x + ref_attention_module(dims, lw, x, len(tokens))
            x = ref_mlp_module(dims, lw, x)
        return F.linear(ref_norm(x, t(W.glob("final_norm")), dims["norm_eps"]), t(W.glob("lm_head")))
    assert np.abs(got - broken(dims, W, toks).numpy()).max() > 1e-3


# ---------------------------------------------------------------------------
# Pin (2): the hand-unrolled ladder recurrence.
# ---------------------------------------------------------------------------
def _unrolled(dims, W, toks, inputs_of):
    """x_k = x_{k-1} + h_k(x_{inputs_of[k]}), written out module by module."""
    xs = [t(W.glob("embed"))[torch.as_tensor(toks, dtype=torch.long)]]
    for k in range(1, 2 * dims["n_layers"] + 1):
        lw = W.layer((k - 1) // 2)
        x_in = xs[inputs_of[k]]
        h = ref_attention_module(dims, lw, x_in, len(toks)) if k % 2 else ref_mlp_module(dims, lw, x_in)
        xs.append(xs[k - 1] + h)
    return F.linear(ref_norm(xs[-1], t(W.glob("final_norm")), dims["norm_eps"]), t(W.glob("lm_head")))


def test_two_layer_ladder_matches_hand_unrolled():
    # x1 = x0 + A1(x0); x2 = x1 + M1(x0); x3 = x2 + A2(x1); x4 = x3 + M2(x2)
    dims = small_dims(n_layers=2, n_standard_layers=0)
    W = random_weights(dims, 3)
    toks = np.array([7, 7, 30, 2, 88, 61])
    got = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True)[0]
    want = _unrolled(dims, W, toks, {1: 0, 2: 0, 3: 1, 4: 2}).numpy()
    close(got, want)
    # and it is not the standard model
    std = _unrolled(dims, W, toks, {1: 0, 2: 1, 3: 2, 4: 3}).numpy()
    assert np.abs(got - std).max() > 1e-3


@pytest.mark.parametrize("strict", [False, True])
def test_hybrid_boundary_matches_hand_unrolled(strict):
    # lower layer standard, two ladder layers above it
    dims = small_dims(n_layers=3, n_standard_layers=1)
    W = random_weights(dims, 4)
    toks = np.array([5, 9, 12, 50, 3])
    got = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True, strict_boundary=strict)[0]
    inputs = {1: 0, 2: 1, 3: 1 if strict else 2, 4: 2, 5: 3, 6: 4}
    close(got, _unrolled(dims, W, toks, inputs).numpy())


# ---------------------------------------------------------------------------
# Pin (3): zeroed module weights give the identity stream.
# ---------------------------------------------------------------------------
def test_zero_modules_give_identity_stream():
    dims = dict(TINY)
    zero = lambda name, layer, a: np.zeros_like(a) if name in ("wo", "w_down") else a
    W = O.synthetic_weights(dims, dtype=np.float64, transform=zero)
    toks = synth.tokens(16, dims["vocab"])
    logits, hist = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True, return_stream=True)
    assert np.array_equal(hist[0][-1], hist[0][0])
    # closed form: logits = W_lm n(E[tok]; g_f)
    E = synth.bf16_bits_to_f32(synth.gen_tensor(dims, "embed")).reshape(dims["vocab"], -1).astype(np.float64)
    Wlm = synth.bf16_bits_to_f32(synth.gen_tensor(dims, "lm_head")).reshape(dims["vocab"], -1).astype(np.float64)
    x = E[toks]
    n = x / np.sqrt((x ** 2).sum(-1, keepdims=True) / x.shape[1] + dims["norm_eps"])
    close(logits[0], n @ Wlm.T, 1e-12)


# ---------------------------------------------------------------------------
# Zeroed W_o or W_down: the stale input equals the fresh one, so ladder == standard bitwise.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kind", ["wo", "w_down"])
def test_zero_output_projection_makes_ladder_standard(kind):
    dims = dict(TINY)
    zero = lambda name, layer, a: np.zeros_like(a) if name == kind else a
    W = O.synthetic_weights(dims, transform=zero)
    toks = synth.tokens(16, dims["vocab"])
    lad = O.forward(dict(dims, n_standard_layers=0), W, [toks], [O.SeqCache()], all_positions=True)[0]
    std = O.forward(dict(dims, n_standard_layers=dims["n_layers"]), W, [toks], [O.SeqCache()],
                    all_positions=True)[0]
    assert np.array_equal(lad, std)


# ---------------------------------------------------------------------------
# Pin (4): decode with the KV cache equals re-running prefill.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("nstd", [0, 1])
def test_cached_decode_equals_prefill_rerun(nstd):
    dims = small_dims(n_layers=2, n_standard_layers=nstd)
    W = random_weights(dims, 5)
    toks = np.array([4, 8, 15, 16, 23, 42, 11, 19, 77])
    P = 5
    logits, caches = O.prefill(dims, W, [toks[:P]])
    rerun = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True)[0]
    close(logits[0], rerun[P - 1], 1e-12)
    for p in range(P, len(toks)):
        step = O.decode_step(dims, W, toks[p:p + 1], caches)
        close(step[0], rerun[p], 1e-12)
    # and against the independent full-recompute block when all layers are standard
    if nstd == dims["n_layers"]:
        close(rerun, ref_standard_forward(dims, W, toks).numpy())


def test_cached_decode_equals_independent_unrolled_ladder():
    dims = small_dims(n_layers=2, n_standard_layers=0)
    W = random_weights(dims, 6)
    toks = np.array([9, 1, 4, 33, 2, 70, 70])
    _, caches = O.prefill(dims, W, [toks[:3]])
    for p in range(3, len(toks)):
        got = O.decode_step(dims, W, toks[p:p + 1], caches)[0]
        want = _unrolled(dims, W, toks[:p + 1], {1: 0, 2: 0, 3: 1, 4: 2}).numpy()[-1]
        close(got, want)


# ---------------------------------------------------------------------------
# Parallel-block model (the comparison model of the pages' 70B table, read as
# the usual parallel attention + MLP layer).
# ---------------------------------------------------------------------------
def ref_parallel_forward(dims, W, tokens):
    """Textbook parallel layer: x <- x + Attn(n_a(x)) + MLP(n_m(x))."""
    x = t(W.glob("embed"))[torch.as_tensor(tokens, dtype=torch.long)]
    for l in range(dims["n_layers"]):
        lw = W.layer(l)
        x = x + ref_attention_module(dims, lw, x, len(tokens)) + ref_mlp_module(dims, lw, x)
    return F.linear(ref_norm(x, t(W.glob("final_norm")), dims["norm_eps"]), t(W.glob("lm_head")))


def test_parallel_block_matches_textbook_and_unrolled():
    dims = small_dims(n_layers=3, n_standard_layers=0)
    W = random_weights(dims, 11)
    toks = np.array([3, 14, 15, 92, 65, 35, 89])
    got = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True, parallel=True)[0]
    close(got, ref_parallel_forward(dims, W, toks).numpy())
    close(got, _unrolled(dims, W, toks, {1: 0, 2: 0, 3: 2, 4: 2, 5: 4, 6: 4}).numpy())
    # it is neither the standard nor the ladder model
    lad = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True)[0]
    std = O.forward(dict(dims, n_standard_layers=3), W, [toks], [O.SeqCache()], all_positions=True)[0]
    assert np.abs(got - lad).max() > 1e-3 and np.abs(got - std).max() > 1e-3


def test_parallel_block_special_cases():
    dims = dict(TINY)
    toks = synth.tokens(16, dims["vocab"])
    # one layer: the ladder layer above x_{-1} := x_0 is a parallel block, bitwise
    one = dict(dims, n_layers=1)
    W1 = O.synthetic_weights(one)
    a = O.forward(one, W1, [toks], [O.SeqCache()], all_positions=True, parallel=True)[0]
    b = O.forward(one, W1, [toks], [O.SeqCache()], all_positions=True)[0]
    assert np.array_equal(a, b)
    # a zero attention output or a zero MLP output makes the parallel block standard, bitwise
    for kind in ("wo", "w_down"):
        zero = lambda name, layer, arr, kind=kind: np.zeros_like(arr) if name == kind else arr
        W = O.synthetic_weights(dims, transform=zero)
        par = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True, parallel=True)[0]
        std = O.forward(dict(dims, n_standard_layers=dims["n_layers"]), W, [toks], [O.SeqCache()],
                        all_positions=True)[0]
        assert np.array_equal(par, std), kind


def test_parallel_cached_decode_equals_prefill_rerun():
    dims = small_dims(n_layers=2, n_standard_layers=0)
    W = random_weights(dims, 12)
    toks = np.array([4, 8, 15, 16, 23, 42, 11, 19])
    P = 4
    logits, caches = O.prefill(dims, W, [toks[:P]], parallel=True)
    rerun = O.forward(dims, W, [toks], [O.SeqCache()], all_positions=True, parallel=True)[0]
    close(logits[0], rerun[P - 1], 1e-12)
    for p in range(P, len(toks)):
        step = O.decode_step(dims, W, toks[p:p + 1], caches, parallel=True)
        close(step[0], rerun[p], 1e-12)


# ---------------------------------------------------------------------------
# Causality and batch independence
# ---------------------------------------------------------------------------
def test_causality_and_batch_independence():
    dims = small_dims(n_layers=2)
    W = random_weights(dims, 7)
    a = np.array([1, 2, 3, 4, 5, 6, 7, 8])
    b = a.copy()
    b[5] = 60
    la = O.forward(dims, W, [a], [O.SeqCache()], all_positions=True)[0]
    lb = O.forward(dims, W, [b], [O.SeqCache()], all_positions=True)[0]
    assert np.array_equal(la[:5], lb[:5])
    assert np.abs(la[5:] - lb[5:]).max() > 1e-6
    # a ragged batch gives each sequence the logits it gets alone
    c = np.array([30, 31, 32])
    both = O.forward(dims, W, [a, c], [O.SeqCache(), O.SeqCache()])
    alone = O.forward(dims, W, [c], [O.SeqCache()])
    assert np.array_equal(both[1], alone[0])
    close(both[0], la[-1], 1e-12)


# ---------------------------------------------------------------------------
# Sub-steps against closed forms and brute force
# ---------------------------------------------------------------------------
def test_rmsnorm_constant_vector():
    for c in (0.5, 3.0, -2.0):
        x = np.full((1, 32), c)
        g = np.linspace(0.5, 1.5, 32)
        eps = 1e-5
        close(O.rmsnorm(x, g, eps)[0], np.sign(c) * g / np.sqrt(1 + eps / c ** 2), 1e-14)


def test_rmsnorm_matches_library():
    rng = np.random.default_rng(0)
    x, g = rng.standard_normal((5, 48)), rng.standard_normal(48)
    close(O.rmsnorm(x, g, 1e-5), ref_norm(t(x), t(g), 1e-5).numpy(), 1e-13)


@pytest.mark.parametrize("interleaved", [True, False])
def test_rope_properties(interleaved):
    rng = np.random.default_rng(1)
    hd, theta = 16, 10000.0
    x = rng.standard_normal((6, 3, hd))
    pos = np.arange(6)
    cos, sin = O.rope_tables(pos, hd, theta, np.float64)
    r = O.apply_rope(x, cos, sin, interleaved)
    # identity at p = 0, rotations preserve norms
    close(r[0], x[0], 1e-15)
    close(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1), 1e-13)
    # q(p).k(p') depends only on p - p'
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    def rot(v, p):
        c, s = O.rope_tables(np.array([p]), hd, theta, np.float64)
        return O.apply_rope(v[None, None, :], c, s, interleaved)[0, 0]
    close(rot(q, 7) @ rot(k, 3), rot(q, 14) @ rot(k, 10), 1e-12)
    # matches rotation by complex multiplication
    close(r, ref_rope(t(x), 0, theta, interleaved).numpy(), 1e-13)


def test_rope_angle_closed_form():
    # pair j of a unit vector at position p lands at (cos(p theta^(-2j/hd)), sin(...))
    hd = 64
    x = np.zeros((1, 1, hd))
    x[0, 0, 0] = 1.0          # pair 0: frequency 1
    x[0, 0, 32] = 1.0         # pair 16: frequency 10000^(-1/2) = 0.01
    c, s = O.rope_tables(np.array([100]), hd, 10000.0, np.float64)
    r = O.apply_rope(x, c, s, True)[0, 0]
    close([r[0], r[1]], [math.cos(100.0), math.sin(100.0)], 1e-12)
    close([r[32], r[33]], [math.cos(1.0), math.sin(1.0)], 1e-12)


def test_attention_brute_force_and_special_cases():
    rng = np.random.default_rng(2)
    T, nq, nkv, hd = 5, 4, 2, 3
    q, k, v = rng.standard_normal((T, nq, hd)), rng.standard_normal((T, nkv, hd)), rng.standard_normal((T, nkv, hd))
    pos = np.arange(T)
    got = O.causal_gqa_attention(q, k, v, pos, pos)
    for ti in range(T):
        for h in range(nq):
            kh = h // 2
            w = [math.exp(sum(q[ti, h, i] * k[s, kh, i] for i in range(hd)) / math.sqrt(hd)) for s in range(ti + 1)]
            z = sum(w)
            want = [sum(w[s] * v[s, kh, i] for s in range(ti + 1)) / z for i in range(hd)]
            close(got[ti, h], want, 1e-12)
    # T = 1 returns v; nkv = nq is multi-head attention (checked against the library)
    close(O.causal_gqa_attention(q[:1], k[:1], v[:1], pos[:1], pos[:1])[0], v[0][[0, 0, 1, 1]], 1e-15)
    k4, v4 = rng.standard_normal((T, nq, hd)), rng.standard_normal((T, nq, hd))
    mha = O.causal_gqa_attention(q, k4, v4, pos, pos)
    lib = F.scaled_dot_product_attention(t(q).transpose(0, 1), t(k4).transpose(0, 1), t(v4).transpose(0, 1),
                                         is_causal=True).transpose(0, 1).numpy()
    close(mha, lib, 1e-13)


def test_silu():
    z = np.array([0.0, 1.0, -1.0, 30.0, -800.0])
    s = O.silu(z)
    assert s[0] == 0.0
    close(s[1:3], [1 / (1 + math.exp(-1)), -1 / (1 + math.e)], 1e-15)
    assert abs(s[3] - 30.0) < 1e-9 and s[4] == 0.0


def test_module_input_index_table():
    # all ladder: module k reads x_{max(k-2, 0)}
    assert [O.module_input_index(k, 0) for k in range(1, 7)] == [0, 0, 1, 2, 3, 4]
    # all standard
    assert [O.module_input_index(k, 3) for k in range(1, 7)] == [0, 1, 2, 3, 4, 5]
    # hybrid with 2 standard layers (b = 4)
    assert [O.module_input_index(k, 2) for k in range(1, 9)] == [0, 1, 2, 3, 4, 4, 5, 6]
    assert [O.module_input_index(k, 2, True) for k in range(1, 9)] == [0, 1, 2, 3, 3, 4, 5, 6]
    # parallel blocks: both modules of layer l read x_{2l}
    assert [O.module_input_index(k, 0, parallel=True) for k in range(1, 7)] == [0, 0, 2, 2, 4, 4]


def test_kv_slot_and_pool_offset():
    bt = np.array([7, 2, 5])
    assert O.kv_slot(bt, 0, 64) == (7, 0)
    assert O.kv_slot(bt, 63, 64) == (7, 63)
    assert O.kv_slot(bt, 64, 64) == (2, 0)
    assert O.kv_slot(bt, 130, 64) == (5, 2)
    # offsets enumerate the pool [L][pages][2][nkv][page][hd] densely in row-major order
    L, P, nkv, ps, hd = 2, 3, 2, 4, 5
    seen = np.zeros(L * P * 2 * nkv * ps * hd, dtype=int)
    for l in range(L):
        for p in range(P):
            for kv in range(2):
                for h in range(nkv):
                    for o in range(ps):
                        off = O.kv_pool_offset(nkv, hd, P, ps, l, p, kv, h, o)
                        seen[off:off + hd] += 1
    assert (seen == 1).all()
    assert O.kv_pool_offset(nkv, hd, P, ps, 1, 2, 1, 1, 3) == np.ravel_multi_index((1, 2, 1, 1, 3, 0), (L, P, 2, nkv, ps, hd))


# ---------------------------------------------------------------------------
# The oracle's own rounding is far below the parity tolerance.
# ---------------------------------------------------------------------------
def test_fp32_oracle_error_is_small():
    dims = dict(TINY)
    toks = [synth.tokens(16, dims["vocab"])]
    l32, _ = O.prefill(dims, O.synthetic_weights(dims, dtype=np.float32), toks)
    l64, _ = O.prefill(dims, O.synthetic_weights(dims, dtype=np.float64), toks)
    assert np.abs(l32 - l64).max() < 1e-4


def test_tiny_greedy_matches_golden():
    import json, os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_greedy.json")
    g = json.load(open(path))
    dims = dict(TINY)
    toks, logits, _ = O.greedy_generate(dims, O.synthetic_weights(dims), [synth.tokens(16, dims["vocab"])], 8)
    assert toks[0].tolist() == g["tokens"]
    assert np.allclose(logits[:, 0, :8], np.array(g["logits_head"]), atol=1e-5)


# ---------------------------------------------------------------------------
# Sampling (temperature / top-k exponential race)
# ---------------------------------------------------------------------------
def test_sampling_mix_matches_published_splitmix64():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "splitmix64.json")))
    gamma = int(g["gamma"], 16)
    for i, want in enumerate(g["outputs_from_state_0"]):
        z = ((i + 1) * gamma) & (2 ** 64 - 1)  # the generator's state after i + 1 steps
        assert O.splitmix64_mix(z) == int(want, 16)
        assert int(O.splitmix64_mix(np.array([z], dtype=np.uint64))[0]) == int(want, 16)


def test_sampling_uniforms_are_exact_and_uniform():
    u = O.sample_uniforms(seed=7, row=1, pos=33, n=200000)
    assert u.min() > 0.0 and u.max() < 1.0
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)  # exact in fp32
    hist = np.histogram(u, bins=20, range=(0, 1))[0]
    assert np.all(np.abs(hist / len(u) - 0.05) < 0.003)
    # different rows and positions give different streams
    assert not np.array_equal(u[:100], O.sample_uniforms(7, 2, 33, 100))
    assert not np.array_equal(u[:100], O.sample_uniforms(7, 1, 34, 100))


def _chi2(counts, probs):
    n = counts.sum()
    e = n * probs
    m = e > 0
    assert np.all(counts[~m] == 0)
    return ((counts[m] - e[m]) ** 2 / e[m]).sum(), int(m.sum()) - 1


@pytest.mark.parametrize("T,k", [(1.0, 0), (0.7, 4), (1.6, 2)])
def test_sampling_distribution_is_softmax_of_the_top_k(T, k):
    """Draws over many positions follow softmax(l / T) restricted to the k
    largest logits: a chi-square test (threshold far in the tail, p ~ 1e-6),
    which a sign flip of the noise, l * T for l / T or an off-by-one top-k set
    all fail."""
    l = np.array([1.2, -0.3, 0.8, 2.0, 0.0, -1.5, 0.5])
    V = len(l)
    N = 30000
    counts = np.zeros(V)
    for pos in range(N):
        counts[O.sample_token(l, T, k, seed=5, row=0, pos=pos)] += 1
    keep = np.ones(V, bool) if k <= 0 else l >= np.sort(l)[V - k]
    p = np.where(keep, np.exp(l / T - (l / T).max()), 0.0)
    p /= p.sum()
    stat, dof = _chi2(counts, p)
    # chi-square tail: dof <= 6 -> p = 1e-6 at about 35
    assert stat < 35.0, (stat, dof, counts / N, p)


def test_sampling_special_cases():
    rng = np.random.default_rng(9)
    l = rng.standard_normal(1000)
    l[417] = 5.0
    for pos in range(20):
        assert O.sample_token(l, 1.0, 1, seed=3, row=2, pos=pos) == 417       # top-1 is greedy
        assert O.sample_token(l, 1e-9, 0, seed=3, row=2, pos=pos) == 417      # T -> 0 is greedy
        assert O.sample_token(l, 0.0, 50, seed=3, row=2, pos=pos) == 417      # T = 0: argmax
        t = O.sample_token(l, 2.0, 10, seed=3, row=2, pos=pos)
        assert l[t] >= np.sort(l)[-10]                                          # inside the top-10
    # ties at the pivot: every logit equal to the k-th largest stays a candidate
    l2 = np.array([3.0, 1.0, 1.0, 1.0, 0.0])
    seen = {O.sample_token(l2, 5.0, 2, seed=1, row=0, pos=p) for p in range(400)}
    assert seen == {0, 1, 2, 3}


# ---------------------------------------------------------------------------
# Rotary frequency scaling (Llama-3.1 rule)
# ---------------------------------------------------------------------------
SCALING = {"factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0, "original_max_position": 8192}


def test_rope_scaling_regimes_and_continuity():
    hd, theta = 128, 500000.0
    f = O.rope_inv_freq(hd, theta)
    g = O.rope_inv_freq(hd, theta, SCALING)
    w = 2 * np.pi / f
    L = SCALING["original_max_position"]
    hi, lo = w < L / 4.0, w > L / 1.0
    assert hi.any() and lo.any() and (~hi & ~lo).any()       # all three regimes occur at this shape
    assert np.array_equal(g[hi], f[hi])                       # short wavelengths untouched
    assert np.allclose(g[lo], f[lo] / 8.0, rtol=0, atol=0)    # long wavelengths divided by the factor
    mid = ~hi & ~lo
    # in between, the ratio g / f falls from 1 towards 1 / factor as the wavelength grows
    r = g / f
    assert np.all((r[mid] < 1.0) & (r[mid] > 1.0 / 8.0))
    assert np.all(np.diff(r) <= 0)
    # the interpolation weight is affine in 1 / wavelength: r = 1/8 + (7/8) s with
    # s = (L / w - 1) / 3, so (r - 1/8) * w is affine in w ... checked through
    # three mid-band points (collinearity of (1/w, r))
    x, y = 1.0 / w[mid], r[mid]
    if len(x) >= 3:
        slope = (y[1:] - y[:-1]) / (x[1:] - x[:-1])
        assert np.allclose(slope, slope[0], rtol=1e-9)
    # scaled frequencies are still decreasing in j (wavelengths increasing)
    assert np.all(np.diff(g) < 0)


def test_rope_scaling_factor_one_is_identity():
    hd, theta = 64, 10000.0
    ident = dict(SCALING, factor=1.0)
    assert np.allclose(O.rope_inv_freq(hd, theta, ident), O.rope_inv_freq(hd, theta), rtol=1e-15, atol=0)
    # no scaling dict: exactly the unscaled angles
    c0, s0 = O.rope_tables(np.arange(5), hd, theta, np.float64)
    c1, s1 = O.rope_tables(np.arange(5), hd, theta, np.float64, None)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
