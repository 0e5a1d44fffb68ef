"""Helpers shared by the GPU parity tests: build a model through the C ABI on the
seeded weights, run the oracle on the same inputs, and compare."""
import functools

import numpy as np
import torch

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import ladder, synth

# Logit tolerance against the fp32 oracle: bf16 weights, fp32 accumulation.
MAX_ABS = 3e-2
REL_L2 = 1e-2
BF16_NAN = 0x7FC0


def small_dims(**over):
    d = dict(synth.PRESETS["tiny"])
    d.update(over)
    return d


@functools.lru_cache(maxsize=4)
def _oracle_weights_cached(key):
    dims = dict(key)
    return O.synthetic_weights(dims)


def oracle_weights(dims, transform=None, keep_layers=True):
    if transform is None and keep_layers:
        # the weights depend on the shapes only (not on e.g. the rotary scaling)
        return _oracle_weights_cached(tuple(sorted((k, v) for k, v in dims.items() if not isinstance(v, dict))))
    return O.synthetic_weights(dims, transform=transform, keep_layers=keep_layers)


def gpu_weights(dims, transform=None, dtype="fp16"):
    return ladder.synthetic_weights(dims, device="cuda", transform=transform, dtype=dtype)


def make_model(dims, weights=None, **kw):
    if weights is None:
        weights = gpu_weights(dims)
    return ladder.LadderModel(dims, weights, **kw)


def compare_logits(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite logits"
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {err:.3e} rel-L2 {rel:.3e}"
    return err, rel


def prompts_for(lens, vocab, seed=synth.PROMPT_SEED):
    return [synth.tokens(n, vocab, seed=seed, stream=b) for b, n in enumerate(lens)]


def packed(prompts):
    return torch.from_numpy(np.concatenate(prompts).astype(np.int32)).cuda()


def check_greedy(gpu_tokens, oracle_logits, err_bound):
    """Greedy tokens must be the oracle's argmax unless the oracle's top-2
    margin is inside the arithmetic's error bound; then the GPU token must be
    one of the oracle's near-maximal candidates.  Returns the indices decided
    by that near-tie rule (an empty list: every token was checked for identity)."""
    ties = []
    for s, (tok, lg) in enumerate(zip(gpu_tokens, oracle_logits)):
        best = int(np.argmax(lg))
        srt = np.sort(lg)
        margin = srt[-1] - srt[-2]
        if margin > err_bound:
            assert tok == best, f"row {s}: token {tok} != oracle {best} (margin {margin:.3e})"
        else:
            ties.append(s)
            assert lg[tok] >= srt[-1] - err_bound, f"row {s}: token {tok} not a near-tie candidate"
    return ties
