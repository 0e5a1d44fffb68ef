"""The seeded input generator: known-answer SplitMix64 outputs, distribution,
chunking and rounding.  It feeds both the CUDA path and the oracle."""
import json
import os

import numpy as np

from ladder_residual_transformer_gb300 import synth


def test_splitmix64_known_answers():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "splitmix64.json")))
    gamma = int(g["gamma"], 16)
    for i, want in enumerate(g["outputs_from_state_0"]):
        assert synth.mix64((i * gamma) & (2 ** 64 - 1)) == int(want, 16)


def test_normal_statistics_and_rounding():
    dims = synth.PRESETS["1.2b"]
    bits = synth.gen_tensor(dims, "wq", 3, count=1 << 20)
    w = synth.bf16_bits_to_f32(bits).astype(np.float64)
    assert abs(w.mean()) < 1e-4
    assert abs(w.std() - 0.02) < 2e-4
    # Irwin-Hall of 8 uniforms: bounded at sqrt(3 * 8) standard deviations
    assert np.abs(w).max() <= 0.02 * np.sqrt(24) * 1.01
    # every value is a bf16 (low 16 fp32 bits zero) and symmetric around zero
    assert abs((w > 0).mean() - 0.5) < 0.01
    # the fp32 scale maps the centred sum's standard deviation to 0.02
    var_sum = 8 * (65536.0 ** 2 - 1) / 12
    assert abs(synth.normal_scale(0.02) * np.sqrt(var_sum) - 0.02) < 1e-8


def test_chunks_match_whole_tensor():
    dims = synth.PRESETS["tiny"]
    whole = synth.gen_tensor(dims, "w_gate", 1)
    parts = [synth.gen_tensor(dims, "w_gate", 1, offset=o, count=min(5000, whole.size - o))
             for o in range(0, whole.size, 5000)]
    assert np.array_equal(np.concatenate(parts), whole)


def test_tensors_differ_and_are_layer_count_independent():
    a = synth.gen_tensor(synth.PRESETS["tiny"], "wq", 0)
    b = synth.gen_tensor(synth.PRESETS["tiny"], "wq", 1)
    c = synth.gen_tensor(synth.PRESETS["tiny"], "wk", 0)
    assert not np.array_equal(a, b) and not np.array_equal(a[: c.size], c)
    dims3 = dict(synth.PRESETS["tiny"], n_layers=3)
    assert np.array_equal(synth.gen_tensor(dims3, "wq", 0), a)


def test_norm_gains_are_one_and_tied_head():
    dims = synth.PRESETS["1.2b"]
    assert (synth.gen_tensor(dims, "attn_norm", 0) == 0x3F80).all()
    assert np.array_equal(synth.gen_tensor(dims, "lm_head", count=4096), synth.gen_tensor(dims, "embed", count=4096))


def test_tokens():
    t = synth.tokens(100000, 1024)
    assert t.min() >= 0 and t.max() < 1024
    assert abs(t.mean() - 511.5) < 5
    assert np.array_equal(synth.tokens(10, 1024, offset=5), t[5:15])
    assert not np.array_equal(synth.tokens(16, 1024, stream=1), t[:16])


def test_param_counts_match_named_sizes():
    assert abs(synth.param_count(synth.PRESETS["1.2b"]) / 1e9 - 1.236) < 0.01
    assert abs(synth.param_count(synth.PRESETS["8b-hybrid"]) / 1e9 - 8.03) < 0.01
    assert abs(synth.param_count(synth.PRESETS["70b"]) * 2 / 1e9 - 141.1) < 0.2


def test_f32_widening_matches_bf16_bits():
    dims = synth.PRESETS["tiny"]
    for name, layer in (("wq", 1), ("embed", -1), ("mlp_norm", 0)):
        a = synth.gen_tensor_f32(dims, name, layer)
        b = synth.bf16_bits_to_f32(synth.gen_tensor(dims, name, layer)).reshape(a.shape)
        assert np.array_equal(a, b)
