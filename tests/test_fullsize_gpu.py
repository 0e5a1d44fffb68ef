"""Full-size workloads on the GPU.

8B hybrid (32 layers, lower 16 standard) against the oracle at full depth; the
70B shapes (d_model 8192, 64 q / 8 kv heads of 128, SwiGLU 28672) with 4 of
their 80 layers against the oracle; and the full 80-layer 70B model (141 GB of
weights resident on the GPU) through properties that hold at any size: decode
with the KV cache agrees with re-running prefill on the extended prompt, and
repeated runs give identical logits.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import ladder, synth

from gpu_common import compare_logits, gpu_weights, make_model, packed, prompts_for

pytestmark = pytest.mark.gpu


def run_tf(model, prompts, feed, graph=True):
    s = torch.cuda.Stream()
    out = []
    with torch.cuda.stream(s):
        model.set_mode(graph=graph)
        lg, _ = model.prefill(packed(prompts), [len(p) for p in prompts])
        out.append(lg.cpu().numpy())
        tok = torch.empty(len(prompts), dtype=torch.int32, device="cuda")
        for i in range(feed.shape[1]):
            tok.copy_(torch.from_numpy(feed[:, i].astype(np.int32)))
            lg, _ = model.decode_step(tok)
            out.append(lg.cpu().numpy())
    s.synchronize()
    return np.stack(out)


def test_device_generator_matches_host_generator():
    dims = synth.PRESETS["1.2b"]
    for name, layer in (("wq", 0), ("w_down", 15), ("embed", -1)):
        n = int(np.prod(synth.tensor_shape(dims, name)))
        raw = torch.empty(n, dtype=torch.int16, device="cuda")
        synth.gen_tensor_device(dims, name, layer, raw.data_ptr())
        torch.cuda.synchronize()
        got = raw.cpu().numpy().view(np.uint16)
        take = slice(0, 1 << 22)
        assert np.array_equal(got[take], synth.gen_tensor(dims, name, layer, count=1 << 22))
        tail = synth.gen_tensor(dims, name, layer, offset=n - 4096, count=4096)
        assert np.array_equal(got[n - 4096:], tail)


@pytest.mark.slow
def test_full_size_8b_hybrid():
    dims = dict(synth.PRESETS["8b-hybrid"])
    lens = [256, 96]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(2, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    gw = gpu_weights(dims)
    model = make_model(dims, gw, max_batch=2, max_seq=512, max_prefill_tokens=sum(lens))
    got = run_tf(model, prompts, feed)
    model.close()
    del gw, model
    torch.cuda.empty_cache()
    want, _ = O.teacher_forced_decode(dims, O.synthetic_weights(dims), prompts, feed)
    # Relative L2 is held to 1e-2.  The max-abs bound is 3e-2, or 1.15x the error
    # of an exactly rounded fp16-activation pipeline on these very inputs when
    # that floor is higher (tests/golden/fp16_floor.py writes it from the oracle:
    # 3.18e-2 for these 32 random layers, so no 16-bit implementation can meet 3e-2).
    floor = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fp16_floor_8b_hybrid.json")))
    max_abs = max(3e-2, 1.15 * floor["max_abs"])
    for s in range(3):
        err = np.abs(got[s] - want[s]).max()
        rel = np.linalg.norm(got[s] - want[s]) / np.linalg.norm(want[s])
        print(f"8B hybrid step {s}: max-abs {err:.3e} rel-L2 {rel:.3e} (fp16 floor {floor['max_abs']:.3e})")
        assert np.isfinite(got[s]).all()
        assert err <= max_abs and rel <= 1e-2, (s, err, rel)


@pytest.mark.slow
def test_70b_shapes_four_layers():
    dims = dict(synth.PRESETS["70b"], n_layers=4)
    lens = [64]
    prompts = prompts_for(lens, dims["vocab"])
    feed = synth.tokens(2, dims["vocab"], seed=synth.DECODE_SEED)[None, :]
    gw = gpu_weights(dims)
    model = make_model(dims, gw, max_batch=1, max_seq=128, max_prefill_tokens=64)
    got = run_tf(model, prompts, feed)
    model.close()
    del gw, model
    torch.cuda.empty_cache()
    want, _ = O.teacher_forced_decode(dims, O.synthetic_weights(dims), prompts, feed)
    for s in range(3):
        compare_logits(got[s], want[s], f"70B shapes step {s}")


@pytest.mark.slow
def test_full_70b_cached_decode_agrees_with_prefill_and_is_deterministic():
    dims = dict(synth.PRESETS["70b"])
    gw = gpu_weights(dims)
    prompt = synth.tokens(34, dims["vocab"])
    model = make_model(dims, gw, max_batch=1, max_seq=64, max_prefill_tokens=64)
    feed = prompt[None, 32:34]
    a = run_tf(model, [prompt[:32]], feed)
    model.reset()
    b = run_tf(model, [prompt[:32]], feed)
    assert np.array_equal(a, b)
    assert np.isfinite(a).all()
    model.reset()
    full = run_tf(model, [prompt], np.zeros((1, 0), dtype=np.int32))
    # Logits after feeding tokens 32 and 33 equal the last-position logits of
    # prefilling all 34.  Both sides are 16-bit-operand computations, each within
    # the oracle tolerance of the true function, so their difference is bounded
    # by the sum of the two bounds.
    err = np.abs(a[2] - full[0]).max()
    rel = np.linalg.norm(a[2] - full[0]) / np.linalg.norm(full[0])
    assert err <= 2 * 3e-2 and rel <= 2 * 1e-2, (err, rel)
    model.close()
