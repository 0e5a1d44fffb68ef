"""Checkpoint loading on the CPU: the safetensors reader and writer, the config
mapping, and the rotary row reordering.

The independent side of the reordering test is the oracle run on the file's own
tensors with the half-split rotary pairing (``rope_interleaved=0``, pinned
against a textbook block built from torch routines in test_oracle_pins.py).  The
loaded, reordered weights must give the same logits with the interleaved
pairing the library computes.
"""
import json
import struct

import numpy as np
import pytest
import torch

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import checkpoint as C
from ladder_residual_transformer_gb300 import synth


def bf16_bits(a):
    """Round fp32 values to bf16 (nearest even) and return the bits (finite inputs)."""
    b = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# The file format
# ---------------------------------------------------------------------------
def test_reads_a_hand_assembled_file(tmp_path):
    """A file put together byte by byte: three dtypes, offsets not in name order,
    a metadata entry, a header padded with spaces."""
    f32 = struct.pack("<6f", 1.5, -2.0, 0.25, 3.0, 4.0, -0.5)
    b16 = struct.pack("<4H", 0x3F80, 0xC000, 0x0000, 0xBE00)  # 1, -2, 0, -0.125
    f16 = struct.pack("<2e", 0.5, -1.0)
    hdr = {"z_f32": {"dtype": "F32", "shape": [2, 3], "data_offsets": [0, 24]},
           "a_bf16": {"dtype": "BF16", "shape": [4], "data_offsets": [28, 36]},
           "m_f16": {"dtype": "F16", "shape": [2], "data_offsets": [24, 28]},
           "__metadata__": {"format": "pt"}}
    text = json.dumps(hdr).encode() + b"   "
    p = tmp_path / "x.safetensors"
    p.write_bytes(struct.pack("<Q", len(text)) + text + f32 + f16 + b16)
    st = C.SafetensorsFile(str(p))
    assert sorted(st.names()) == ["a_bf16", "m_f16", "z_f32"]
    assert st.metadata == {"format": "pt"}
    dt, a = st.get("z_f32")
    assert dt == "F32" and a.shape == (2, 3)
    assert np.array_equal(a, np.array([[1.5, -2.0, 0.25], [3.0, 4.0, -0.5]], np.float32))
    dt, a = st.get("a_bf16")
    assert dt == "BF16" and np.array_equal(synth.bf16_bits_to_f32(np.asarray(a)), [1.0, -2.0, 0.0, -0.125])
    dt, a = st.get("m_f16")
    assert dt == "F16" and np.array_equal(a, np.array([0.5, -1.0], np.float16))


def test_writer_round_trip(tmp_path):
    g = torch.Generator().manual_seed(3)
    tensors = {
        "w.bf16": torch.randn(5, 7, generator=g).to(torch.bfloat16),
        "w.f16": torch.randn(3, generator=g).to(torch.float16),
        "w.f32": torch.randn(2, 2, 2, generator=g),
        "n.f32": np.linspace(-1, 1, 9, dtype=np.float32),
        "b.bits": ("BF16", np.array([0x3F80, 0x4000, 0x8000], np.uint16)),
        "e.empty": torch.zeros(0, 4, dtype=torch.bfloat16),
    }
    p = str(tmp_path / "rt.safetensors")
    C.write_safetensors(p, tensors, metadata={"k": 1})
    raw = open(p, "rb").read()
    n = struct.unpack("<Q", raw[:8])[0]
    assert n % 8 == 0
    hdr = json.loads(raw[8:8 + n])
    assert hdr.pop("__metadata__") == {"k": "1"}
    offs = [hdr[k]["data_offsets"] for k in sorted(hdr)]
    assert offs[0][0] == 0 and all(a[1] == b[0] for a, b in zip(offs, offs[1:]))
    assert offs[-1][1] == len(raw) - 8 - n
    st = C.SafetensorsFile(p)
    _, a = st.get("w.bf16")
    assert np.array_equal(np.asarray(a), tensors["w.bf16"].view(torch.int16).numpy().view(np.uint16))
    _, a = st.get("w.f16")
    assert np.array_equal(a, tensors["w.f16"].numpy())
    _, a = st.get("w.f32")
    assert np.array_equal(a, tensors["w.f32"].numpy())
    _, a = st.get("n.f32")
    assert np.array_equal(a, tensors["n.f32"])
    _, a = st.get("b.bits")
    assert np.array_equal(a, [0x3F80, 0x4000, 0x8000])
    dt, a = st.get("e.empty")
    assert dt == "BF16" and a.shape == (0, 4)


def _file(tmp_path, hdr, data=b"", hdr_len=None):
    text = json.dumps(hdr).encode() if isinstance(hdr, dict) else hdr
    p = tmp_path / "bad.safetensors"
    p.write_bytes(struct.pack("<Q", len(text) if hdr_len is None else hdr_len) + text + data)
    return str(p)


@pytest.mark.parametrize("case", ["short", "hdr_len", "not_json", "offsets", "size", "dtype", "entry"])
def test_rejects_malformed_files(tmp_path, case):
    ok = {"t": {"dtype": "F32", "shape": [2], "data_offsets": [0, 8]}}
    if case == "short":
        p = tmp_path / "s.safetensors"
        p.write_bytes(b"\x01\x00")
        p = str(p)
    elif case == "hdr_len":
        p = _file(tmp_path, ok, b"\x00" * 8, hdr_len=10 ** 6)
    elif case == "not_json":
        p = _file(tmp_path, b"{not json", b"")
    elif case == "offsets":
        p = _file(tmp_path, ok, b"\x00" * 4)
    elif case == "size":
        p = _file(tmp_path, {"t": {"dtype": "F32", "shape": [3], "data_offsets": [0, 8]}}, b"\x00" * 8)
    elif case == "dtype":
        p = _file(tmp_path, {"t": {"dtype": "I64", "shape": [1], "data_offsets": [0, 8]}}, b"\x00" * 8)
    else:
        p = _file(tmp_path, {"t": {"dtype": "F32"}}, b"")
    with pytest.raises(ValueError):
        C.SafetensorsFile(p)


# ---------------------------------------------------------------------------
# Config mapping
# ---------------------------------------------------------------------------
LLAMA31_8B = {  # the architecture fields of a Llama-3.1-8B config
    "hidden_size": 4096, "num_hidden_layers": 32, "num_attention_heads": 32, "num_key_value_heads": 8,
    "intermediate_size": 14336, "vocab_size": 128256, "rms_norm_eps": 1e-5, "rope_theta": 500000.0,
    "hidden_act": "silu", "tie_word_embeddings": False, "attention_bias": False, "mlp_bias": False,
    "rope_scaling": {"rope_type": "llama3", "factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
                     "original_max_position_embeddings": 8192},
}


def test_dims_from_hf_config():
    d = C.dims_from_hf_config(LLAMA31_8B, 16)
    ref = synth.PRESETS["8b-hybrid"]
    for k in ("n_layers", "n_standard_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "ffn_dim",
              "vocab", "tie_embeddings", "rope_interleaved", "norm_eps"):
        assert d[k] == ref[k], k
    assert d["rope_theta"] == 500000.0
    assert d["rope_scaling"] == dict(factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0,
                                     original_max_position=8192)
    mha = dict(LLAMA31_8B, num_key_value_heads=None, rope_scaling=None, tie_word_embeddings=True, head_dim=64)
    d = C.dims_from_hf_config(mha, 0)
    assert d["n_kv_heads"] == 32 and d["head_dim"] == 64 and d["tie_embeddings"] == 1 and "rope_scaling" not in d
    d = C.dims_from_hf_config(dict(LLAMA31_8B, rope_scaling={"rope_type": "default"}), 32)
    assert "rope_scaling" not in d and d["n_standard_layers"] == 32
    # a 16-layer, 2048-wide model with tied embeddings has the shapes of the 1.2B workload
    small = dict(LLAMA31_8B, hidden_size=2048, num_hidden_layers=16, intermediate_size=8192, head_dim=64,
                 tie_word_embeddings=True)
    d = C.dims_from_hf_config(small, 0)
    ref = synth.PRESETS["1.2b"]
    assert all(d[k] == ref[k] for k in ("n_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "ffn_dim",
                                        "vocab", "tie_embeddings"))


@pytest.mark.parametrize("over,nstd", [({"hidden_act": "gelu"}, 0), ({"attention_bias": True}, 0),
                                       ({"mlp_bias": True}, 0), ({"rope_scaling": {"rope_type": "yarn"}}, 0),
                                       ({}, 33), ({}, -1)])
def test_dims_rejects_what_the_library_does_not_compute(over, nstd):
    with pytest.raises(ValueError):
        C.dims_from_hf_config(dict(LLAMA31_8B, **over), nstd)


# ---------------------------------------------------------------------------
# Rotary row order
# ---------------------------------------------------------------------------
def test_row_order_written_out():
    assert C.half_split_to_interleaved_rows(2, 8).tolist() == [0, 4, 1, 5, 2, 6, 3, 7, 8, 12, 9, 13, 10, 14, 11, 15]
    assert C.half_split_to_interleaved_rows(1, 2).tolist() == [0, 1]


def test_row_order_turns_half_split_rotation_into_interleaved():
    """Rotating z_j = x_j + i x_{j+hd/2} (half split) and then reordering equals
    reordering and then rotating z_j = x_{2j} + i x_{2j+1} (interleaved):
    complex rotation written with torch, at several positions."""
    H, hd, theta = 3, 16, 10000.0
    x = torch.randn(5, H, hd, dtype=torch.float64, generator=torch.Generator().manual_seed(1))
    f = theta ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    rot = torch.polar(torch.ones(5, hd // 2, dtype=torch.float64), torch.outer(torch.arange(5.0, 10.0), f))[:, None]
    z = torch.complex(x[..., :hd // 2], x[..., hd // 2:]) * rot
    half = torch.cat([z.real, z.imag], -1).reshape(5, H * hd)
    perm = torch.from_numpy(C.half_split_to_interleaved_rows(H, hd))
    xp = x.reshape(5, H * hd)[:, perm].reshape(5, H, hd)
    zi = torch.view_as_complex(xp.reshape(5, H, hd // 2, 2).contiguous()) * rot
    inter = torch.view_as_real(zi).reshape(5, H * hd)
    assert torch.allclose(half[:, perm], inter, atol=1e-14, rtol=0)


# ---------------------------------------------------------------------------
# Whole checkpoints
# ---------------------------------------------------------------------------
def hf_checkpoint(tmp_path, dims, *, tied=False, shards=2, rope_scaling=None, seed=5, drop=(), std=0.2,
                  gain_std=0.3):
    """Random bf16 tensors under the Hugging Face names (gains near 1, weights with
    std 0.2 by default so that every module matters), written as ``shards`` files
    plus an index and a config.json.  Returns {name: bf16 bits}."""
    rng = np.random.default_rng(seed)
    names = [("embed", -1), ("final_norm", -1)] + ([] if tied else [("lm_head", -1)])
    names += [(k, l) for l in range(dims["n_layers"]) for k in synth.LAYER_KINDS]
    bits = {}
    for kind, l in names:
        shape = synth.tensor_shape(dims, kind)
        v = 1.0 + gain_std * rng.standard_normal(shape) if kind in synth.NORM_KINDS else std * rng.standard_normal(shape)
        bits[C.hf_name(kind, l)] = bf16_bits(v)
    keep = [n for n in sorted(bits) if n not in drop]
    wm = {}
    for s in range(shards):
        part = keep[s::shards]
        fn = f"model-{s + 1:05d}-of-{shards:05d}.safetensors"
        C.write_safetensors(str(tmp_path / fn), {n: ("BF16", bits[n]) for n in part})
        wm.update({n: fn for n in part})
    (tmp_path / "model.safetensors.index.json").write_text(json.dumps({"metadata": {}, "weight_map": wm}))
    cfg = {"hidden_size": dims["d_model"], "num_hidden_layers": dims["n_layers"],
           "num_attention_heads": dims["n_q_heads"], "num_key_value_heads": dims["n_kv_heads"],
           "head_dim": dims["head_dim"], "intermediate_size": dims["ffn_dim"], "vocab_size": dims["vocab"],
           "rms_norm_eps": dims["norm_eps"], "rope_theta": dims["rope_theta"], "hidden_act": "silu",
           "tie_word_embeddings": tied, "rope_scaling": rope_scaling}
    (tmp_path / "config.json").write_text(json.dumps(cfg))
    return bits


def oracle_from_bits(dims, bits):
    """fp64 oracle weights straight from the file's bf16 bits (no reordering)."""
    def source(kind, layer):
        return synth.bf16_bits_to_f32(bits[C.hf_name(kind, layer)]).astype(np.float64)
    return O.OracleWeights(dims, source, dtype=np.float64)


def oracle_from_loaded(dims, w):
    def source(kind, layer):
        t = w[kind] if layer < 0 else w["layers"][layer][kind]
        return t.float().numpy().astype(np.float64)
    return O.OracleWeights(dims, source, dtype=np.float64)


DIMS = dict(n_layers=3, n_standard_layers=1, d_model=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96,
            vocab=97, rope_theta=10000.0, norm_eps=1e-5, rope_interleaved=1, tie_embeddings=0)
SCALING = {"rope_type": "llama3", "factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
           "original_max_position_embeddings": 64}


@pytest.mark.parametrize("tied", [False, True])
def test_loaded_model_equals_the_half_split_model(tmp_path, tied):
    """fp64 oracle: the file's tensors with half-split rotary pairs vs the loaded
    (reordered) tensors with interleaved pairs, hybrid layout, Llama-3.1 rotary
    scaling, all positions of a 12-token prompt plus one cached decode step."""
    bits = hf_checkpoint(tmp_path, DIMS, tied=tied, rope_scaling=SCALING)
    dims, w = C.load_llama(str(tmp_path), n_standard_layers=1, device="cpu", dtype="bf16")
    assert dims["tie_embeddings"] == int(tied) and (w["lm_head"] is None) == tied
    assert dims["rope_scaling"]["original_max_position"] == 64
    # storage: bf16 bits kept; q rows reordered, v rows not
    hd = DIMS["head_dim"]
    wq = w["layers"][2]["wq"].view(torch.int16).numpy().view(np.uint16)
    fq = bits[C.hf_name("wq", 2)]
    assert np.array_equal(wq[hd + 2 * 3], fq[hd + 3]) and np.array_equal(wq[hd + 2 * 3 + 1], fq[hd + hd // 2 + 3])
    assert np.array_equal(w["layers"][0]["wv"].view(torch.int16).numpy().view(np.uint16), bits[C.hf_name("wv", 0)])
    ref_dims = dict(dims, rope_interleaved=0)
    toks = np.array([5, 90, 17, 17, 3, 0, 64, 41, 8, 2, 77, 13])
    ref_c, got_c = O.SeqCache(), O.SeqCache()
    want = O.forward(ref_dims, oracle_from_bits(ref_dims, bits), [toks], [ref_c], all_positions=True)[0]
    W = oracle_from_loaded(dims, w)
    got = O.forward(dims, W, [toks], [got_c], all_positions=True)[0]
    assert np.abs(got - want).max() <= 1e-10 * np.abs(want).max()
    want1 = O.forward(ref_dims, oracle_from_bits(ref_dims, bits), [np.array([33])], [ref_c])
    got1 = O.forward(dims, W, [np.array([33])], [got_c])
    assert np.abs(got1 - want1).max() <= 1e-10 * np.abs(want1).max()


def test_skipping_the_reordering_changes_the_model(tmp_path):
    """Sensitivity of the test above: loading half-split rows as if they were
    interleaved gives a different model."""
    bits = hf_checkpoint(tmp_path, DIMS)
    dims, w = C.load_llama(str(tmp_path), n_standard_layers=1, device="cpu", dtype="bf16",
                           rope_layout="interleaved")
    ref_dims = dict(dims, rope_interleaved=0)
    toks = np.array([5, 90, 17, 17, 3, 0, 64, 41])
    want = O.forward(ref_dims, oracle_from_bits(ref_dims, bits), [toks], [O.SeqCache()])
    got = O.forward(dims, oracle_from_loaded(dims, w), [toks], [O.SeqCache()])
    assert np.abs(got - want).max() > 1e-3


def test_fp16_storage_rounds_to_nearest(tmp_path):
    bits = hf_checkpoint(tmp_path, DIMS, shards=1)
    _, w = C.load_llama(str(tmp_path), n_standard_layers=0, device="cpu", dtype="fp16")
    got = w["layers"][1]["w_up"]
    assert got.dtype == torch.float16
    want = torch.from_numpy(synth.bf16_bits_to_f32(bits[C.hf_name("w_up", 1)])).to(torch.float16)
    assert torch.equal(got, want)


def test_missing_or_misshapen_tensors(tmp_path):
    hf_checkpoint(tmp_path, DIMS, drop=("lm_head.weight",))
    with pytest.raises(ValueError, match="lm_head"):
        C.load_llama(str(tmp_path), n_standard_layers=0, device="cpu")
    cfg = json.loads((tmp_path / "config.json").read_text())
    with pytest.raises(ValueError, match="shape"):
        C.load_llama(str(tmp_path), n_standard_layers=0, device="cpu",
                     config=dict(cfg, intermediate_size=128, tie_word_embeddings=True))
    with pytest.raises(ValueError, match="rope_layout"):
        C.load_llama(str(tmp_path), n_standard_layers=0, device="cpu", rope_layout="neox")
