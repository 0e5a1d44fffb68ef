"""Thin Python binding of libladder.so (declared in include/ladder.h).

Argument marshalling only: every step of the forward pass runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  If the
library is missing or cannot be built, importing the model raises: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

LADDER_OK = 0
LADDER_ERR_INVALID = -1
LADDER_ERR_CUDA = -2
LADDER_ERR_CAPACITY = -3
LADDER_ERR_UNSUPPORTED = -4

RESIDUAL_CONFIG = 0
RESIDUAL_STANDARD = 1
RESIDUAL_PARALLEL = 2
FLAG_DECODE_GRAPH = 1
FLAG_NO_PDL = 2
FLAG_ALL_LOGITS = 4
FLAG_FAST_PREFILL = 8

# Entry points declared in include/ladder.h, with (restype, argtypes).
_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_pi32 = ctypes.POINTER(ctypes.c_int32)


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "n_standard_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab")] + [
        ("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float)] + [(n, ctypes.c_int32) for n in (
            "tie_embeddings", "rope_interleaved", "shard_k", "page_size", "max_batch", "max_seq",
            "max_prefill_tokens", "strict_boundary", "weight_dtype")] + [
        ("rope_scale_factor", ctypes.c_float), ("rope_low_freq_factor", ctypes.c_float),
        ("rope_high_freq_factor", ctypes.c_float), ("rope_original_max_pos", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("final_norm", _vp), ("lm_head", _vp)] + [
        (n, ctypes.POINTER(_vp)) for n in (
            "attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")]


_SIGNATURES = {
    "ladder_query_sizes": (_i32, [ctypes.POINTER(Config), ctypes.POINTER(_sz), ctypes.POINTER(_sz)]),
    "ladder_create": (_i32, [ctypes.POINTER(Config), ctypes.POINTER(Weights), _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "ladder_destroy": (None, [_vp]),
    "ladder_set_mode": (_i32, [_vp, ctypes.c_int, ctypes.c_int]),
    "ladder_kv_create": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp, ctypes.POINTER(_vp)]),
    "ladder_kv_destroy": (None, [_vp]),
    "ladder_kv_set_pages": (_i32, [_vp, _pi32, _vp]),
    "ladder_kv_reset": (_i32, [_vp, _vp]),
    "ladder_kv_seq_len": (_i32, [_vp, _i32]),
    "ladder_prefill": (_i32, [_vp, _vp, _vp, _pi32, _i32, _vp, _vp, _vp]),
    "ladder_decode_step": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _vp]),
    "ladder_get_device_error": (_i32, [_vp, _vp, _pi32]),
    "ladder_last_launch_count": (_i32, [_vp]),
    "ladder_probe_begin": (_i32, [_vp, ctypes.c_int, _i32]),
    "ladder_probe_end": (_i32, [_vp, _pi32, ctypes.POINTER(_f32)]),
    "ladder_attention_decode_scratch_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "ladder_attention_decode": (_i32, [_vp, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _i32,
                                       _vp, _vp, _sz, _vp]),
    "ladder_attention_decode_noalloc": (_i32, [_vp, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32,
                                               _i32, _vp, _vp]),
    "ladder_timeline_begin": (_i32, [_vp, _i32, _vp]),
    "ladder_timeline_end": (_i32, [_vp, _i32, _pi32, _vp, _vp, _vp, _vp]),
    "ladder_set_sampling": (_i32, [_vp, _f32, _i32, ctypes.c_uint64]),
    "ladder_sample": (_i32, [_vp, _i32, _i32, _f32, _i32, ctypes.c_uint64, _vp, _i32, _vp, _vp]),
    "ladder_last_error": (ctypes.c_char_p, []),
}

STATIC_SCRATCH_BYTES = 8 << 20  # LADDER_STATIC_SCRATCH_BYTES

PROBE_CLASSES = {"qkv": 0, "attn": 1, "out": 2, "gateup": 3, "down": 4, "lmhead": 5, "reduce": 6}


def lib(build_if_missing: bool = True):
    """The loaded library; builds it first when it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libladder.so not found at {path}; run __graft_entry__.build()")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


class LadderError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libladder error {code}: {msg}")
        self.code = code


def check(rc: int):
    if rc != LADDER_OK:
        raise LadderError(rc, lib().ladder_last_error().decode())


DTYPES = {"bf16": 0, "fp16": 1}


def make_config(dims: dict, *, max_batch: int, max_seq: int, max_prefill_tokens: int | None = None,
                page_size: int = 64, shard_k: int = 1, strict_boundary: int = 0, dtype: str = "fp16") -> Config:
    return Config(
        n_layers=dims["n_layers"], n_standard_layers=dims["n_standard_layers"], d_model=dims["d_model"],
        n_q_heads=dims["n_q_heads"], n_kv_heads=dims["n_kv_heads"], head_dim=dims["head_dim"],
        ffn_dim=dims["ffn_dim"], vocab=dims["vocab"], rope_theta=dims["rope_theta"], norm_eps=dims["norm_eps"],
        tie_embeddings=dims.get("tie_embeddings", 0), rope_interleaved=dims.get("rope_interleaved", 1),
        shard_k=shard_k, page_size=page_size, max_batch=max_batch, max_seq=max_seq,
        max_prefill_tokens=max_prefill_tokens if max_prefill_tokens is not None else max_batch * max_seq,
        strict_boundary=strict_boundary, weight_dtype=DTYPES[dtype],
        **_rope_scaling_fields(dims.get("rope_scaling")))


def _rope_scaling_fields(sc: dict | None) -> dict:
    if not sc:
        return {}
    return dict(rope_scale_factor=float(sc["factor"]), rope_low_freq_factor=float(sc["low_freq_factor"]),
                rope_high_freq_factor=float(sc["high_freq_factor"]),
                rope_original_max_pos=int(sc["original_max_position"]))


def query_sizes(cfg: Config) -> tuple[int, int]:
    ws, page = _sz(0), _sz(0)
    check(lib().ladder_query_sizes(ctypes.byref(cfg), ctypes.byref(ws), ctypes.byref(page)))
    return ws.value, page.value


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def synthetic_weights(dims: dict, device="cuda", seed: int = 0, transform=None, dtype: str = "fp16") -> dict:
    """Random-init weights of the seeded generator, produced on the device.

    The device twin of the generator writes the same bf16 bits as the host code
    (tests check this); with dtype="fp16" each tensor is then converted on the
    device (round to nearest even), which is exact for 2^-17 <= |w| <= 65504,
    i.e. for all but a few hundredths of a percent of N(0, 0.02) values, whose
    error is below 3e-8.  ``transform(name, layer, np_bits) -> np_bits`` edits
    a tensor's bf16 bits on the host first (small tensors only).
    Returns {"embed": T, "final_norm": T, "lm_head": T or None, "layers": [dict], "dtype": str}.
    """
    from . import synth

    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    stream = torch.cuda.current_stream(device)

    def make(name, layer):
        shape = synth.tensor_shape(dims, name)
        n = int(np.prod(shape))
        raw = torch.empty(n, dtype=torch.int16, device=device)
        if transform is not None:
            bits = np.ascontiguousarray(transform(name, layer, synth.gen_tensor(dims, name, layer, seed=seed)))
            raw.copy_(torch.from_numpy(bits.view(np.int16)))
        elif name in synth.NORM_KINDS:
            raw.fill_(0x3F80)
        else:
            synth.gen_tensor_device(dims, name, layer, raw.data_ptr(), seed=seed, stream_ptr=stream.cuda_stream)
        t = raw.view(torch.bfloat16) if tdt == torch.bfloat16 else raw.view(torch.bfloat16).to(tdt)
        return t.view(shape)

    out = {"embed": make("embed", -1), "final_norm": make("final_norm", -1),
           "lm_head": None if dims.get("tie_embeddings") else make("lm_head", -1), "layers": [],
           "dtype": dtype}
    for l in range(dims["n_layers"]):
        out["layers"].append({k: make(k, l) for k in synth.LAYER_KINDS})
    torch.cuda.synchronize(device)
    return out


def _kv_dtype(t: torch.Tensor) -> int:
    """C-ABI code of a KV tensor's 16-bit type (int16 views count as bf16)."""
    return DTYPES["fp16"] if t.dtype == torch.float16 else DTYPES["bf16"]


def attention_decode(q: torch.Tensor, kv_layer: torch.Tensor, block_table: torch.Tensor, positions: torch.Tensor,
                     n_kv_heads: int, head_dim: int, page_size: int, max_position: int, scale: float | None = None,
                     out: torch.Tensor | None = None, scratch: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Standalone decode attention through the C ABI (see ladder_attention_decode)."""
    B = positions.numel()
    n_q = q.shape[-1] // head_dim
    if scale is None:
        scale = head_dim ** -0.5
    if out is None:
        out = torch.empty(B, n_q * head_dim, dtype=torch.float32, device=q.device)
    need = lib().ladder_attention_decode_scratch_bytes(B, n_q, head_dim, max_position)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=q.device)
    check(lib().ladder_attention_decode(q.data_ptr(), kv_layer.data_ptr(), _kv_dtype(kv_layer), block_table.data_ptr(),
                                        block_table.shape[-1], positions.data_ptr(), B, n_q, n_kv_heads, head_dim,
                                        page_size, scale, max_position, out.data_ptr(), scratch.data_ptr(),
                                        scratch.numel() * scratch.element_size(), _stream_handle(stream)))
    return out


def attention_decode_noalloc(q: torch.Tensor, kv_layer: torch.Tensor, block_table: torch.Tensor,
                             positions: torch.Tensor, n_kv_heads: int, head_dim: int, page_size: int,
                             max_position: int, out: torch.Tensor, scale: float | None = None, stream=None):
    """Decode attention through the entry point that allocates nothing
    (ladder_attention_decode_noalloc): its scratch is a static device array."""
    B = positions.numel()
    n_q = q.shape[-1] // head_dim
    if scale is None:
        scale = head_dim ** -0.5
    check(lib().ladder_attention_decode_noalloc(q.data_ptr(), kv_layer.data_ptr(), _kv_dtype(kv_layer),
                                                block_table.data_ptr(),
                                                block_table.shape[-1], positions.data_ptr(), B, n_q, n_kv_heads,
                                                head_dim, page_size, scale, max_position, out.data_ptr(),
                                                _stream_handle(stream)))
    return out


def sample(logits: torch.Tensor, positions: torch.Tensor, temperature: float, top_k: int = 0, seed: int = 0,
           pos_offset: int = 0, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Temperature / top-k sampling of each row of device fp32 logits [B, V]
    through the C ABI (see ladder_sample); positions: device int32 [B]."""
    B, V = logits.shape
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=logits.device)
    check(lib().ladder_sample(logits.data_ptr(), B, V, float(temperature), int(top_k), int(seed) & (2 ** 64 - 1),
                              positions.data_ptr(), int(pos_offset), out.data_ptr(), _stream_handle(stream)))
    return out


class LadderModel:
    """A model over device weights plus its paged KV cache, driven through the C ABI.

    Pages are assigned contiguously by default: sequence b owns pages
    page_order[b*pps : (b+1)*pps], pps = ceil(max_seq / page_size).
    """

    def __init__(self, dims: dict, weights: dict, *, max_batch: int, max_seq: int,
                 max_prefill_tokens: int | None = None, page_size: int = 64, strict_boundary: int = 0,
                 page_order=None, kv_fill_bits: int | None = None, stream=None, shard_k: int = 1):
        self.dims = dict(dims)
        self.weights = weights
        self.cfg = make_config(dims, max_batch=max_batch, max_seq=max_seq, max_prefill_tokens=max_prefill_tokens,
                               page_size=page_size, strict_boundary=strict_boundary, shard_k=shard_k,
                               dtype=weights.get("dtype", "bf16"))
        L = lib()
        ws_bytes, self.page_bytes = query_sizes(self.cfg)
        dev = weights["embed"].device
        self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.max_batch, self.max_seq, self.page_size = max_batch, max_seq, page_size
        self.pages_per_seq = (max_seq + page_size - 1) // page_size
        self.num_pages = max_batch * self.pages_per_seq
        self.kv_pool = torch.empty(self.num_pages * self.page_bytes, dtype=torch.uint8, device=dev)
        if kv_fill_bits is not None:
            self.kv_pool.view(torch.int16).fill_(kv_fill_bits - 65536 if kv_fill_bits >= 32768 else kv_fill_bits)
        self.block_table = torch.full((max_batch, self.pages_per_seq), -1, dtype=torch.int32, device=dev)
        self.seq_lens = torch.zeros(max_batch, dtype=torch.int32, device=dev)

        layers = weights["layers"]
        self._ptr_arrays = {}
        for k in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"):
            arr = (_vp * len(layers))(*[layers[l][k].data_ptr() for l in range(len(layers))])
            self._ptr_arrays[k] = arr
        w = Weights(embed=weights["embed"].data_ptr(), final_norm=weights["final_norm"].data_ptr(),
                    lm_head=weights["lm_head"].data_ptr() if weights.get("lm_head") is not None else None,
                    **{k: ctypes.cast(v, ctypes.POINTER(_vp)) for k, v in self._ptr_arrays.items()})
        s = _stream_handle(stream)
        self._m = _vp()
        check(L.ladder_create(ctypes.byref(self.cfg), ctypes.byref(w), self.workspace.data_ptr(), ws_bytes, s,
                              ctypes.byref(self._m)))
        self._kv = _vp()
        check(L.ladder_kv_create(self._m, self.kv_pool.data_ptr(), self.num_pages, self.pages_per_seq,
                                 self.block_table.data_ptr(), self.seq_lens.data_ptr(), ctypes.byref(self._kv)))
        order = np.arange(self.num_pages, dtype=np.int32) if page_order is None else np.asarray(page_order, np.int32)
        self.host_table = np.ascontiguousarray(order.reshape(max_batch, self.pages_per_seq))
        self.set_pages(self.host_table, stream)
        self.reset(stream)

    # -- cache -----------------------------------------------------------
    def set_pages(self, host_table: np.ndarray, stream=None):
        t = np.ascontiguousarray(host_table, dtype=np.int32)
        check(lib().ladder_kv_set_pages(self._kv, t.ctypes.data_as(_pi32), _stream_handle(stream)))
        self.host_table = t

    def reset(self, stream=None):
        check(lib().ladder_kv_reset(self._kv, _stream_handle(stream)))

    def seq_len(self, b: int) -> int:
        return lib().ladder_kv_seq_len(self._kv, b)

    # -- modes -----------------------------------------------------------
    def set_mode(self, standard: bool = False, graph: bool = False, pdl: bool = True, parallel: bool = False,
                 all_logits: bool = False, fast_prefill: bool = False):
        """Residual schedule: as configured (default), every layer standard
        (``standard``), or every layer a parallel attention + MLP block
        (``parallel``); decode launch flags; ``all_logits``: prefill returns the
        logits of every packed position ([sum of lens, vocab]);
        ``fast_prefill``: prefill GEMM activations rounded once to 16 bits
        instead of carried as hi/lo pairs (half the tensor-core work, less
        accurate on deep models; see LADDER_FLAG_FAST_PREFILL)."""
        if standard and parallel:
            raise ValueError("standard and parallel are exclusive")
        flags = (FLAG_DECODE_GRAPH if graph else 0) | (0 if pdl else FLAG_NO_PDL) | (FLAG_ALL_LOGITS if all_logits else 0)
        flags |= FLAG_FAST_PREFILL if fast_prefill else 0
        mode = RESIDUAL_STANDARD if standard else RESIDUAL_PARALLEL if parallel else RESIDUAL_CONFIG
        check(lib().ladder_set_mode(self._m, mode, flags))
        self._standard = standard
        self._parallel = parallel
        self._all_logits = all_logits
        self._fast_prefill = fast_prefill

    def set_sampling(self, temperature: float = 0.0, top_k: int = 0, seed: int = 0):
        """Next-token rule of prefill / decode_step: greedy (temperature <= 0) or
        temperature / top-k sampling with SplitMix64 draws keyed by seed, batch
        row and position (see ladder_set_sampling)."""
        check(lib().ladder_set_sampling(self._m, float(temperature), int(top_k), int(seed) & (2 ** 64 - 1)))

    # -- forward ---------------------------------------------------------
    def prefill(self, tokens: torch.Tensor, lens, logits: torch.Tensor | None = None,
                next_tok: torch.Tensor | None = None, stream=None):
        """tokens: device int32 packed prompts; lens: host list of lengths.
        Logits: [B, vocab] of each last position, or [sum of lens, vocab] of
        every position when set_mode(all_logits=True)."""
        B = len(lens)
        hl = np.ascontiguousarray(lens, dtype=np.int32)
        dev = tokens.device
        if logits is None:
            rows = int(hl.sum()) if getattr(self, "_all_logits", False) else B
            logits = torch.empty(rows, self.dims["vocab"], dtype=torch.float32, device=dev)
        if next_tok is None:
            next_tok = torch.empty(B, dtype=torch.int32, device=dev)
        check(lib().ladder_prefill(self._m, self._kv, tokens.data_ptr(), hl.ctypes.data_as(_pi32), B,
                                   logits.data_ptr(), next_tok.data_ptr(), _stream_handle(stream)))
        return logits, next_tok

    def decode_step(self, tokens: torch.Tensor, logits: torch.Tensor | None = None,
                    next_tok: torch.Tensor | None = None, stream=None):
        """tokens: device int32 [B]; next_tok may be the same tensor as tokens."""
        B = tokens.numel()
        dev = tokens.device
        if logits is None:
            logits = torch.empty(B, self.dims["vocab"], dtype=torch.float32, device=dev)
        if next_tok is None:
            next_tok = torch.empty(B, dtype=torch.int32, device=dev)
        check(lib().ladder_decode_step(self._m, self._kv, tokens.data_ptr(), B, logits.data_ptr(),
                                       next_tok.data_ptr(), _stream_handle(stream)))
        return logits, next_tok

    def generate(self, prompts, n_new: int, stream=None) -> np.ndarray:
        """Greedy generation from host prompts to host tokens [B, n_new + 1].

        The prompt ids go to the device from pinned memory, prefill and n_new
        decode steps run with the greedy token fed back on the device, and the
        generated ids come back to pinned host memory once at the end.
        """
        lens = [len(p) for p in prompts]
        B, total = len(lens), int(sum(lens))
        st = stream if stream is not None else torch.cuda.current_stream()
        dev = self.weights["embed"].device
        key = (B, total, n_new)
        if getattr(self, "_gen_key", None) != key:
            self._gen_key = key
            self._h_prompt = torch.empty(total, dtype=torch.int32, pin_memory=True)
            self._d_prompt = torch.empty(total, dtype=torch.int32, device=dev)
            self._d_tok = torch.empty(B, dtype=torch.int32, device=dev)
            self._d_logits = torch.empty(B, self.dims["vocab"], dtype=torch.float32, device=dev)
            self._d_hist = torch.empty(n_new + 1, B, dtype=torch.int32, device=dev)
            self._h_hist = torch.empty(n_new + 1, B, dtype=torch.int32, pin_memory=True)
        self._h_prompt.numpy()[:] = np.concatenate(prompts).astype(np.int32)
        with torch.cuda.stream(st):
            self.reset(st)
            self._d_prompt.copy_(self._h_prompt, non_blocking=True)
            self.prefill(self._d_prompt, lens, self._d_logits, self._d_tok, st)
            self._d_hist[0].copy_(self._d_tok)
            for i in range(n_new):
                self.decode_step(self._d_tok, self._d_logits, self._d_tok, st)
                self._d_hist[i + 1].copy_(self._d_tok)
            self._h_hist.copy_(self._d_hist, non_blocking=True)
        st.synchronize()
        return self._h_hist.numpy().T.copy()

    def device_error(self, stream=None) -> int:
        code = ctypes.c_int32(0)
        check(lib().ladder_get_device_error(self._m, _stream_handle(stream), ctypes.byref(code)))
        return code.value

    def probe_begin(self, kernel_class: str, max_launches: int = 65536):
        check(lib().ladder_probe_begin(self._m, PROBE_CLASSES[kernel_class], max_launches))

    def probe_end(self) -> tuple[int, float]:
        n, ms = ctypes.c_int32(0), ctypes.c_float(0)
        check(lib().ladder_probe_end(self._m, ctypes.byref(n), ctypes.byref(ms)))
        return n.value, ms.value

    def timeline_begin(self, max_launches: int, stream=None):
        """Arm the launch timeline for the following eager decode steps."""
        check(lib().ladder_timeline_begin(self._m, max_launches, _stream_handle(stream)))
        self._tl_cap = max_launches

    def timeline_end(self) -> list[tuple[int, str, float, float]]:
        """(stream, class name, start ms, end ms) of each recorded launch, in issue order."""
        cap = getattr(self, "_tl_cap", 0)
        st = np.zeros(cap, np.int32)
        cl = np.zeros(cap, np.int32)
        t0 = np.zeros(cap, np.float32)
        t1 = np.zeros(cap, np.float32)
        n = ctypes.c_int32(0)
        check(lib().ladder_timeline_end(self._m, cap, ctypes.byref(n), st.ctypes.data, cl.ctypes.data,
                                        t0.ctypes.data, t1.ctypes.data))
        names = {v: k for k, v in PROBE_CLASSES.items()}
        return [(int(st[i]), names[int(cl[i])], float(t0[i]), float(t1[i])) for i in range(n.value)]

    def last_launch_count(self) -> int:
        return lib().ladder_last_launch_count(self._m)

    def kv_view(self) -> torch.Tensor:
        """The pool in its 16-bit type, [n_layers][num_pages][2][n_kv][page_size][head_dim]."""
        d = self.dims
        t = torch.float16 if self.cfg.weight_dtype == DTYPES["fp16"] else torch.bfloat16
        return self.kv_pool.view(t).view(d["n_layers"], self.num_pages, 2, d["n_kv_heads"], self.page_size,
                                         d["head_dim"])

    def close(self):
        L = lib()
        if getattr(self, "_kv", None):
            L.ladder_kv_destroy(self._kv)
            self._kv = None
        if getattr(self, "_m", None):
            L.ladder_destroy(self._m)
            self._m = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
