"""Seeded synthetic inputs: model dimensions of the named workloads, random-init
bf16 weights and random token ids.

This module is the only code that the CUDA path and the CPU oracle share.  It
holds none of the model's arithmetic; it only says which tensors exist, what
shape they have, and which bits they hold.  The generator itself is the small C
file next to this one (SplitMix64 counters, an Irwin-Hall sum of eight 16-bit
uniforms, round-to-nearest-even to bf16), compiled on first use.

Workloads (Ladder Transformer, Zhang et al., "Ladder-residual: parallelism-aware
architecture for accelerating large model inference with communication
overlapping", arXiv 2501.06589): the 1.2B and 8B/70B shapes are the model sizes
that the paper trains and benchmarks (its inference-speedup table lists 1B, 3B,
8B, 34B, 70B, 176B and 405B); the dimensions themselves are Llama-style.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libladder_synth.so")
_CU_SRC = os.path.join(_HERE, "synth_cuda.cu")
_CU_LIB_PATH = os.path.join(_HERE, "libladder_synth_cuda.so")
_lib = None
_cu_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to its source."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_cuda(force: bool = False) -> str:
    """Compile the device twin of the generator (sm_103a)."""
    if not force and os.path.exists(_CU_LIB_PATH) and os.path.getmtime(_CU_LIB_PATH) >= os.path.getmtime(_CU_SRC):
        return _CU_LIB_PATH
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared", "-Xcompiler", "-fPIC",
           "-o", tmp, _CU_SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _CU_LIB_PATH)
    return _CU_LIB_PATH


def _load_cuda():
    global _cu_lib
    with _lock:
        if _cu_lib is None:
            lib = ctypes.CDLL(build_cuda())
            lib.synth_normal_bf16_device.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                                     ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
            lib.synth_normal_bf16_device.restype = ctypes.c_int
            _cu_lib = lib
    return _cu_lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, u32, f32 = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_float
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, f32, ctypes.c_void_p]
            lib.synth_normal_bf16.restype = None
            lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, f32, ctypes.c_void_p]
            lib.synth_normal_f32.restype = None
            lib.synth_tokens.argtypes = [u64, u64, u64, u64, u32, ctypes.c_void_p]
            lib.synth_tokens.restype = None
            lib.synth_mix64.argtypes = [u64]
            lib.synth_mix64.restype = u64
            lib.synth_normal_scale.argtypes = [f32]
            lib.synth_normal_scale.restype = f32
            lib.synth_stream_key.argtypes = [u64, u64]
            lib.synth_stream_key.restype = u64
            _lib = lib
    return _lib


# ---------------------------------------------------------------------------
# Named workloads.  Keys are model dimensions only; the run shapes (prompt
# length, decode steps, batch) sit in RUNS.
# ---------------------------------------------------------------------------
_COMMON = dict(rope_theta=10000.0, norm_eps=1e-5, rope_interleaved=1)

PRESETS = {
    "tiny": dict(n_layers=2, n_standard_layers=0, d_model=256, n_q_heads=4, n_kv_heads=2,
                 head_dim=64, ffn_dim=768, vocab=1024, tie_embeddings=0, **_COMMON),
    "1.2b": dict(n_layers=16, n_standard_layers=0, d_model=2048, n_q_heads=32, n_kv_heads=8,
                 head_dim=64, ffn_dim=8192, vocab=128256, tie_embeddings=1, **_COMMON),
    "8b-hybrid": dict(n_layers=32, n_standard_layers=16, d_model=4096, n_q_heads=32, n_kv_heads=8,
                      head_dim=128, ffn_dim=14336, vocab=128256, tie_embeddings=0, **_COMMON),
    "8b-ladder": dict(n_layers=32, n_standard_layers=0, d_model=4096, n_q_heads=32, n_kv_heads=8,
                      head_dim=128, ffn_dim=14336, vocab=128256, tie_embeddings=0, **_COMMON),
    "70b": dict(n_layers=80, n_standard_layers=0, d_model=8192, n_q_heads=64, n_kv_heads=8,
                head_dim=128, ffn_dim=28672, vocab=128256, tie_embeddings=0, **_COMMON),
}

RUNS = {
    "tiny": dict(batch=1, prompt=16, decode_steps=8),
    "1.2b": dict(batch=1, prompt=1024, decode_steps=256),
    "8b-hybrid": dict(batch=4, prompt=4096, decode_steps=4, decode_batches=(1, 16), decode_ctx=2048),
    "8b-ladder": dict(batch=1, prompt=2048, decode_steps=128, shard_k=8),
    "70b": dict(batch=1, prompt=512, decode_steps=4, decode_ctx=2048),
}

INIT_STD = 0.02
WEIGHT_SEED = 0
PROMPT_SEED = 1
DECODE_SEED = 2

# Tensor ids: global tensors use small ids; layer l, kind k uses ((l + 1) << 8) | k,
# so a layer's weights do not depend on how many layers the model has.
_GLOBAL_IDS = {"embed": 1, "final_norm": 2, "lm_head": 3}
LAYER_KINDS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")
_LAYER_IDS = {name: i + 1 for i, name in enumerate(LAYER_KINDS)}
NORM_KINDS = ("attn_norm", "mlp_norm", "final_norm")


def tensor_shape(dims: dict, name: str) -> tuple:
    d, hq, hkv, hd = dims["d_model"], dims["n_q_heads"], dims["n_kv_heads"], dims["head_dim"]
    f, v = dims["ffn_dim"], dims["vocab"]
    return {
        "embed": (v, d), "final_norm": (d,), "lm_head": (v, d),
        "attn_norm": (d,), "wq": (hq * hd, d), "wk": (hkv * hd, d), "wv": (hkv * hd, d),
        "wo": (d, hq * hd), "mlp_norm": (d,), "w_gate": (f, d), "w_up": (f, d), "w_down": (d, f),
    }[name]


def tensor_id(name: str, layer: int = -1) -> int:
    if layer < 0:
        return _GLOBAL_IDS[name]
    return ((layer + 1) << 8) | _LAYER_IDS[name]


def gen_tensor(dims: dict, name: str, layer: int = -1, seed: int = WEIGHT_SEED,
               out: np.ndarray | None = None, offset: int = 0, count: int | None = None) -> np.ndarray:
    """bf16 bits (uint16) of a weight tensor, flattened row-major.

    Norm gains are all ones (bf16 0x3F80).  `offset`/`count` select a slice of
    the flattened tensor so large tensors can be produced in chunks.
    """
    if name == "lm_head" and dims.get("tie_embeddings"):
        name = "embed"
    n_total = int(np.prod(tensor_shape(dims, name)))
    if count is None:
        count = n_total - offset
    if out is None:
        out = np.empty(count, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size >= count
    assert 0 <= offset and offset + count <= n_total
    if name in NORM_KINDS:
        out[:count] = 0x3F80
    else:
        _load().synth_normal_bf16(seed, tensor_id(name, layer), offset, count, INIT_STD,
                                  out.ctypes.data)
    return out[:count]


def gen_tensor_f32(dims: dict, name: str, layer: int = -1, seed: int = WEIGHT_SEED) -> np.ndarray:
    """The same values as gen_tensor, widened exactly to fp32, shaped like the tensor."""
    if name == "lm_head" and dims.get("tie_embeddings"):
        name = "embed"
    shape = tensor_shape(dims, name)
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    if name in NORM_KINDS:
        out[:] = 1.0
    else:
        _load().synth_normal_f32(seed, tensor_id(name, layer), 0, n, INIT_STD, out.ctypes.data)
    return out.reshape(shape)


def tokens(n: int, vocab: int, seed: int = PROMPT_SEED, stream: int = 0, offset: int = 0) -> np.ndarray:
    """n uniform token ids in [0, vocab) for sequence `stream`."""
    out = np.empty(n, dtype=np.int32)
    if n:
        _load().synth_tokens(seed, stream, offset, n, vocab, out.ctypes.data)
    return out


def mix64(z: int) -> int:
    return int(_load().synth_mix64(z))


def normal_scale(std: float = INIT_STD) -> float:
    return float(_load().synth_normal_scale(std))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def param_count(dims: dict) -> int:
    n = 0
    for name in ("embed", "final_norm"):
        n += int(np.prod(tensor_shape(dims, name)))
    if not dims.get("tie_embeddings"):
        n += int(np.prod(tensor_shape(dims, "lm_head")))
    for name in LAYER_KINDS:
        n += dims["n_layers"] * int(np.prod(tensor_shape(dims, name)))
    return n


def gen_tensor_device(dims: dict, name: str, layer: int, out_ptr: int, seed: int = WEIGHT_SEED,
                      stream_ptr: int = 0) -> int:
    """Write the bf16 bits of a weight tensor into device memory at out_ptr
    (the same bits as gen_tensor); returns the element count."""
    if name == "lm_head" and dims.get("tie_embeddings"):
        name = "embed"
    n = int(np.prod(tensor_shape(dims, name)))
    if name in NORM_KINDS:
        raise ValueError("norm gains are constant; fill them directly")
    key = int(_load().synth_stream_key(seed, tensor_id(name, layer)))
    rc = _load_cuda().synth_normal_bf16_device(key, 0, n, normal_scale(INIT_STD), out_ptr, stream_ptr)
    if rc != 0:
        raise RuntimeError(f"device generator launch failed ({rc})")
    return n
