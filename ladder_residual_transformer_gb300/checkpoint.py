"""Llama-family checkpoints in the safetensors format, loaded as ladder weights.

The Ladder Residual paper adapts a pretrained Llama-3.1 model by keeping its
lower layers standard and switching the upper ones to the ladder residual; the
weights are reused as they are ("Ladder Residual: Parallelism-Aware Architecture
for Accelerating Large Model Inference", section 关键设计, hybrid adaptation).
The official code also reads such checkpoints' rotary scaling (its
apply_rope_scaling helper, named in the codewithpapers record "Ladder-residual:
parallelism-aware architecture for accelerating large model inference with
communication overlapping").  So loading a checkpoint means reading its tensors,
mapping their names, and two layout changes.  All of it happens on the host or
as plain copies; the forward pass does not change.

* Rotary pairing.  Checkpoints in the Hugging Face layout order each head's rows
  of W_q and W_k for the half-split pairing, where row j rotates with row
  j + hd/2.  The library rotates interleaved pairs (2j, 2j+1) by the same angle
  p * f_j.  So each head's rows are reordered: new row 2j = old row j, new row
  2j+1 = old row j + hd/2.  Each pair then holds the same two coordinates and
  turns by the same angle, and q.k sums the same products, so the model
  computes the same function.  W_v and W_o are unchanged.
  ``rope_layout="interleaved"`` skips this step for checkpoints already in
  interleaved order.
* Storage type.  bf16, fp16 or fp32 tensors are converted to the library's fp16
  (the default) or bf16 storage; the conversion rounds to nearest even.

The safetensors layout:
* an unsigned little-endian 64-bit header length n;
* n bytes of UTF-8 JSON mapping each tensor name to {"dtype", "shape",
  "data_offsets": [begin, end]}, where the offsets point into the data that
  follows the header;
* an optional "__metadata__" entry of strings inside that JSON;
* then the tensors' bytes, little-endian and row-major.
A sharded checkpoint adds model.safetensors.index.json, whose "weight_map" names
the file of each tensor.
"""
from __future__ import annotations

import json
import os
import struct

import numpy as np
import torch

from . import synth

# safetensors dtype -> (numpy dtype of the stored elements, bytes per element); BF16 is kept as raw bits
_ST_DTYPES = {"BF16": (np.dtype("<u2"), 2), "F16": (np.dtype("<f2"), 2), "F32": (np.dtype("<f4"), 4)}
_TORCH_TO_ST = {torch.bfloat16: "BF16", torch.float16: "F16", torch.float32: "F32"}

# Hugging Face Llama tensor names of the library's weights
HF_GLOBAL = {"embed": "model.embed_tokens.weight", "final_norm": "model.norm.weight", "lm_head": "lm_head.weight"}
HF_LAYER = {
    "attn_norm": "input_layernorm.weight", "wq": "self_attn.q_proj.weight", "wk": "self_attn.k_proj.weight",
    "wv": "self_attn.v_proj.weight", "wo": "self_attn.o_proj.weight", "mlp_norm": "post_attention_layernorm.weight",
    "w_gate": "mlp.gate_proj.weight", "w_up": "mlp.up_proj.weight", "w_down": "mlp.down_proj.weight",
}


def hf_name(kind: str, layer: int = -1) -> str:
    """Checkpoint name of the library weight ``kind`` (of layer ``layer``)."""
    return HF_GLOBAL[kind] if layer < 0 else f"model.layers.{layer}.{HF_LAYER[kind]}"


class SafetensorsFile:
    """One safetensors file: its header parsed and checked, its tensors memory-mapped on demand."""

    def __init__(self, path: str):
        self.path = path
        size = os.path.getsize(path)
        with open(path, "rb") as f:
            head = f.read(8)
            if len(head) != 8:
                raise ValueError(f"{path}: shorter than the 8-byte header length")
            n = struct.unpack("<Q", head)[0]
            if n > size - 8:
                raise ValueError(f"{path}: header length {n} exceeds the file ({size} bytes)")
            try:
                hdr = json.loads(f.read(n).decode("utf-8"))
            except (UnicodeDecodeError, json.JSONDecodeError) as e:
                raise ValueError(f"{path}: header is not JSON: {e}") from None
        if not isinstance(hdr, dict):
            raise ValueError(f"{path}: header is not a JSON object")
        self.data_start = 8 + n
        self.metadata = hdr.pop("__metadata__", None) or {}
        data_len = size - self.data_start
        self.entries: dict[str, tuple[str, tuple, int]] = {}
        for name, e in hdr.items():
            try:
                dt, shape, (begin, end) = e["dtype"], tuple(int(s) for s in e["shape"]), e["data_offsets"]
            except (KeyError, TypeError, ValueError):
                raise ValueError(f"{path}: malformed entry for {name!r}") from None
            if dt not in _ST_DTYPES:
                raise ValueError(f"{path}: {name}: dtype {dt} is not supported (BF16, F16, F32)")
            if any(s < 0 for s in shape) or not (0 <= begin <= end <= data_len):
                raise ValueError(f"{path}: {name}: offsets [{begin}, {end}) outside the data ({data_len} bytes)")
            if end - begin != int(np.prod(shape, dtype=np.int64)) * _ST_DTYPES[dt][1]:
                raise ValueError(f"{path}: {name}: {end - begin} bytes for shape {shape} of {dt}")
            self.entries[name] = (dt, shape, int(begin))

    def __contains__(self, name: str) -> bool:
        return name in self.entries

    def names(self) -> list[str]:
        return list(self.entries)

    def get(self, name: str) -> tuple[str, np.ndarray]:
        """(dtype string, read-only array of the stored elements); BF16 comes as uint16 bits."""
        dt, shape, begin = self.entries[name]
        npdt = _ST_DTYPES[dt][0]
        n = int(np.prod(shape, dtype=np.int64))
        if n == 0:
            return dt, np.zeros(shape, npdt)
        return dt, np.memmap(self.path, dtype=npdt, mode="r", offset=self.data_start + begin, shape=(n,)).reshape(shape)


def write_safetensors(path: str, tensors: dict, metadata: dict | None = None) -> None:
    """Write ``tensors`` (name -> torch tensor of bf16/fp16/fp32, numpy fp16/fp32
    array, or ("BF16", uint16 bits array)) as one safetensors file, in name order,
    with the header padded by spaces to a multiple of 8 bytes."""
    blobs, hdr, off = [], {}, 0
    for name in sorted(tensors):
        t = tensors[name]
        if isinstance(t, tuple):
            dt, a = t
            if dt != "BF16":
                raise ValueError(f"{name}: tuple form is for BF16 bits only")
            a = np.ascontiguousarray(a, dtype="<u2")
            shape, raw = a.shape, a.tobytes()
        elif isinstance(t, torch.Tensor):
            if t.dtype not in _TORCH_TO_ST:
                raise ValueError(f"{name}: torch dtype {t.dtype} is not supported")
            dt, shape = _TORCH_TO_ST[t.dtype], tuple(t.shape)
            c = t.detach().cpu().contiguous().reshape(-1)
            raw = (c.view(torch.int16) if c.element_size() == 2 else c.view(torch.int32)).numpy().astype(
                "<i2" if c.element_size() == 2 else "<i4", copy=False).tobytes()
        else:
            a = np.asarray(t)
            dt = {np.dtype(np.float16): "F16", np.dtype(np.float32): "F32"}.get(a.dtype)
            if dt is None:
                raise ValueError(f"{name}: numpy dtype {a.dtype} is not supported (pass ('BF16', bits) for bf16)")
            shape, raw = a.shape, np.ascontiguousarray(a, dtype=_ST_DTYPES[dt][0]).tobytes()
        hdr[name] = {"dtype": dt, "shape": [int(s) for s in shape], "data_offsets": [off, off + len(raw)]}
        blobs.append(raw)
        off += len(raw)
    if metadata:
        hdr["__metadata__"] = {str(k): str(v) for k, v in metadata.items()}
    text = json.dumps(hdr, separators=(",", ":")).encode("utf-8")
    text += b" " * (-len(text) % 8)
    with open(path, "wb") as f:
        f.write(struct.pack("<Q", len(text)))
        f.write(text)
        for b in blobs:
            f.write(b)


class Checkpoint:
    """A checkpoint directory (config.json plus model.safetensors, or shards listed
    in model.safetensors.index.json, or every *.safetensors file) or one file."""

    def __init__(self, path: str):
        if os.path.isfile(path):
            root, files = os.path.dirname(os.path.abspath(path)), [path]
        else:
            root = path
            index = os.path.join(path, "model.safetensors.index.json")
            if os.path.exists(index):
                with open(index) as f:
                    wm = json.load(f)["weight_map"]
                files = sorted({os.path.join(path, v) for v in wm.values()})
            else:
                files = sorted(os.path.join(path, n) for n in os.listdir(path) if n.endswith(".safetensors"))
            if not files:
                raise FileNotFoundError(f"{path}: no safetensors files")
        cfg_path = os.path.join(root, "config.json")
        self.config = None
        if os.path.exists(cfg_path):
            with open(cfg_path) as f:
                self.config = json.load(f)
        self._where: dict[str, SafetensorsFile] = {}
        for fp in files:
            st = SafetensorsFile(fp)
            for name in st.names():
                if name in self._where:
                    raise ValueError(f"tensor {name} appears in {self._where[name].path} and {fp}")
                self._where[name] = st

    def __contains__(self, name: str) -> bool:
        return name in self._where

    def get(self, name: str) -> tuple[str, np.ndarray]:
        if name not in self._where:
            raise KeyError(f"checkpoint has no tensor {name}")
        return self._where[name].get(name)


def dims_from_hf_config(cfg: dict, n_standard_layers: int) -> dict:
    """Model dimensions of a Hugging Face Llama config.

    ``n_standard_layers`` lower layers keep the standard residual and the rest
    become ladder layers (the paper's hybrid adaptation converts the upper
    half).  Only what the library computes is accepted: SiLU-gated MLPs, no
    biases, and rotary scaling of the Llama-3.1 kind or none.
    """
    if cfg.get("hidden_act", "silu") != "silu":
        raise ValueError(f"hidden_act {cfg.get('hidden_act')!r}: only silu is supported")
    if cfg.get("attention_bias") or cfg.get("mlp_bias"):
        raise ValueError("projection biases are not supported")
    d, nq = int(cfg["hidden_size"]), int(cfg["num_attention_heads"])
    L = int(cfg["num_hidden_layers"])
    if not 0 <= n_standard_layers <= L:
        raise ValueError(f"n_standard_layers {n_standard_layers} outside [0, {L}]")
    dims = dict(
        n_layers=L, n_standard_layers=int(n_standard_layers), d_model=d, n_q_heads=nq,
        n_kv_heads=int(cfg.get("num_key_value_heads") or nq), head_dim=int(cfg.get("head_dim") or d // nq),
        ffn_dim=int(cfg["intermediate_size"]), vocab=int(cfg["vocab_size"]),
        rope_theta=float(cfg.get("rope_theta", 10000.0)), norm_eps=float(cfg["rms_norm_eps"]),
        tie_embeddings=int(bool(cfg.get("tie_word_embeddings", False))), rope_interleaved=1)
    sc = cfg.get("rope_scaling")
    if sc:
        kind = sc.get("rope_type", sc.get("type"))
        if kind == "llama3":
            dims["rope_scaling"] = dict(factor=float(sc["factor"]), low_freq_factor=float(sc["low_freq_factor"]),
                                        high_freq_factor=float(sc["high_freq_factor"]),
                                        original_max_position=int(sc["original_max_position_embeddings"]))
        elif kind != "default":
            raise ValueError(f"rotary scaling {kind!r} is not supported (llama3 or none)")
    return dims


def half_split_to_interleaved_rows(n_heads: int, head_dim: int) -> np.ndarray:
    """Row order that takes a half-split rotary projection to the interleaved one:
    within each head, new row 2j = old row j and new row 2j+1 = old row j + hd/2."""
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    half = head_dim // 2
    per_head = np.empty(head_dim, dtype=np.int64)
    per_head[0::2] = np.arange(half)
    per_head[1::2] = np.arange(half) + half
    return (np.arange(n_heads, dtype=np.int64)[:, None] * head_dim + per_head[None, :]).reshape(-1)


def load_llama(path: str, *, n_standard_layers: int, device="cuda", dtype: str = "fp16",
               rope_layout: str = "half_split", config: dict | None = None) -> tuple[dict, dict]:
    """Read a Llama checkpoint into (dims, weights) for ``LadderModel``.

    The weights dict has the layout of ``ladder.synthetic_weights``: device
    tensors in ``dtype`` ("fp16" or "bf16"), one dict per layer.
    ``rope_layout`` says how the checkpoint pairs rotary coordinates:
    "half_split" (the Hugging Face layout: W_q and W_k rows are reordered) or
    "interleaved" (kept).  ``config`` overrides the checkpoint's config.json.
    """
    if rope_layout not in ("half_split", "interleaved"):
        raise ValueError(f"rope_layout {rope_layout!r}: half_split or interleaved")
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    ck = Checkpoint(path)
    cfg = config if config is not None else ck.config
    if cfg is None:
        raise ValueError(f"{path}: no config.json and no config given")
    dims = dims_from_hf_config(cfg, n_standard_layers)
    rows = {}
    if rope_layout == "half_split":
        rows["wq"] = half_split_to_interleaved_rows(dims["n_q_heads"], dims["head_dim"])
        rows["wk"] = half_split_to_interleaved_rows(dims["n_kv_heads"], dims["head_dim"])

    def fetch(kind: str, layer: int = -1) -> torch.Tensor:
        name = hf_name(kind, layer)
        dt, a = ck.get(name)
        want = synth.tensor_shape(dims, kind)
        if tuple(a.shape) != tuple(want):
            raise ValueError(f"{name}: shape {tuple(a.shape)}, the config implies {want}")
        a = np.array(a[rows[kind]] if kind in rows else a)  # an owned host copy
        host = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "BF16" else torch.from_numpy(a)
        return host.to(device).to(tdt)

    weights = {"embed": fetch("embed"), "final_norm": fetch("final_norm"), "layers": [], "dtype": dtype}
    if dims["tie_embeddings"]:
        weights["lm_head"] = None
    elif HF_GLOBAL["lm_head"] in ck:
        weights["lm_head"] = fetch("lm_head")
    else:
        raise ValueError("the config says the embeddings are not tied, but there is no lm_head.weight")
    for l in range(dims["n_layers"]):
        weights["layers"].append({k: fetch(k, l) for k in synth.LAYER_KINDS})
    return dims, weights
