"""Host-side checks of libladder.so that need no GPU: it builds for sm_103a,
loads, exports every entry point include/ladder.h declares, and validates
configurations before touching a device."""
import ctypes
import os
import re

import pytest

from ladder_residual_transformer_gb300 import ladder, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ladder_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_entry_point():
    L = ladder.lib()
    names = declared_functions()
    assert "ladder_prefill" in names and "ladder_decode_step" in names
    for n in names:
        assert hasattr(L, n), n
    # the binding's signature table covers the header exactly
    assert names == set(ladder._SIGNATURES)


def test_binding_constants_match_the_header():
    """Every enumerator of include/ladder.h that the binding mirrors has the same value."""
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "ladder.h")).read(), flags=re.S)
    enum = {k: int(v) for k, v in re.findall(r"\b(LADDER_[A-Z0-9_]+)\s*=\s*(-?\d+)", text)}
    for name in ("OK", "ERR_INVALID", "ERR_CUDA", "ERR_CAPACITY", "ERR_UNSUPPORTED"):
        assert getattr(ladder, "LADDER_" + name) == enum["LADDER_" + name], name
    for name in ("CONFIG", "STANDARD", "PARALLEL"):
        assert getattr(ladder, "RESIDUAL_" + name) == enum["LADDER_RESIDUAL_" + name], name
    for name in ("DECODE_GRAPH", "NO_PDL", "ALL_LOGITS", "FAST_PREFILL"):
        assert getattr(ladder, "FLAG_" + name) == enum["LADDER_FLAG_" + name], name
    for cls, v in ladder.PROBE_CLASSES.items():
        key = "LADDER_PROBE_" + {"out": "OUT", "gateup": "GATEUP", "lmhead": "LMHEAD"}.get(cls, cls.upper())
        assert enum[key] == v, cls
    assert len(ladder.PROBE_CLASSES) == sum(k.startswith("LADDER_PROBE_") for k in enum)
    assert ladder.DTYPES == {"bf16": enum["LADDER_DTYPE_BF16"], "fp16": enum["LADDER_DTYPE_F16"]}


def cfg(**over):
    dims = dict(synth.PRESETS["tiny"])
    c = ladder.make_config(dims, max_batch=4, max_seq=256)
    for k, v in over.items():
        setattr(c, k, v)
    return c


def test_query_sizes_and_page_bytes():
    ws, page = ladder.query_sizes(cfg())
    d = synth.PRESETS["tiny"]
    assert page == d["n_layers"] * 2 * d["n_kv_heads"] * 64 * d["head_dim"] * 2
    assert ws > 3 * 4 * 256 * d["d_model"] * 4  # three fp32 stream buffers at least


@pytest.mark.parametrize("field,value,code", [
    ("d_model", 300, ladder.LADDER_ERR_INVALID),
    ("head_dim", 96, ladder.LADDER_ERR_UNSUPPORTED),
    ("n_kv_heads", 3, ladder.LADDER_ERR_INVALID),
    ("n_standard_layers", 3, ladder.LADDER_ERR_INVALID),
    ("vocab", 1023, ladder.LADDER_ERR_INVALID),
    ("page_size", 48, ladder.LADDER_ERR_INVALID),
    ("max_batch", 65, ladder.LADDER_ERR_INVALID),
    ("rope_interleaved", 0, ladder.LADDER_ERR_UNSUPPORTED),
    ("norm_eps", 0.0, ladder.LADDER_ERR_INVALID),
])
def test_invalid_configs_are_rejected_on_the_host(field, value, code):
    with pytest.raises(ladder.LadderError) as e:
        ladder.query_sizes(cfg(**{field: value}))
    assert e.value.code == code
    assert ladder.lib().ladder_last_error()


@pytest.mark.parametrize("fields", [
    dict(rope_scale_factor=8.0, rope_low_freq_factor=4.0, rope_high_freq_factor=1.0, rope_original_max_pos=8192),
    dict(rope_scale_factor=8.0, rope_low_freq_factor=0.0, rope_high_freq_factor=4.0, rope_original_max_pos=8192),
    dict(rope_scale_factor=8.0, rope_low_freq_factor=1.0, rope_high_freq_factor=4.0, rope_original_max_pos=0),
])
def test_invalid_rope_scaling_is_rejected(fields):
    with pytest.raises(ladder.LadderError) as e:
        ladder.query_sizes(cfg(**fields))
    assert e.value.code == ladder.LADDER_ERR_INVALID


def test_rope_scaling_off_and_valid_configs_are_accepted():
    ladder.query_sizes(cfg(rope_scale_factor=1.0))
    ladder.query_sizes(cfg(rope_scale_factor=8.0, rope_low_freq_factor=1.0, rope_high_freq_factor=4.0,
                           rope_original_max_pos=8192))


def test_null_arguments_are_rejected_without_a_device():
    L = ladder.lib()
    out = ctypes.c_void_p()
    c = cfg()
    assert L.ladder_create(ctypes.byref(c), None, None, 0, None, ctypes.byref(out)) == ladder.LADDER_ERR_INVALID
    assert out.value is None
    assert L.ladder_decode_step(None, None, None, 1, None, None, None) == ladder.LADDER_ERR_INVALID
    assert L.ladder_prefill(None, None, None, None, 1, None, None, None) == ladder.LADDER_ERR_INVALID
    assert L.ladder_kv_seq_len(None, 0) == -1
    assert L.ladder_last_launch_count(None) == -1
    # entry points added with the sampler, the schedules and the tracing aids
    assert L.ladder_set_sampling(None, 1.0, 0, 0) == ladder.LADDER_ERR_INVALID
    assert L.ladder_set_mode(None, 2, 0) == ladder.LADDER_ERR_INVALID
    assert L.ladder_sample(None, 1, 10, 1.0, 0, 0, None, 0, None, None) == ladder.LADDER_ERR_INVALID
    n = ctypes.c_int32(0)
    assert L.ladder_timeline_begin(None, 16, None) == ladder.LADDER_ERR_INVALID
    assert L.ladder_timeline_end(None, 0, ctypes.byref(n), None, None, None, None) == ladder.LADDER_ERR_INVALID
    assert L.ladder_probe_begin(None, 0, 16) == ladder.LADDER_ERR_INVALID
