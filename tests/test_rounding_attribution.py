"""The rounding-attribution aid of the oracle: its lock-step forward pass is the
oracle's forward pass, rounding nothing changes nothing, and each rounding
point it names moves the logits by a small, nonzero amount."""
import numpy as np

import oracle.ladder_oracle as O
from oracle import rounding_attribution as RA
from ladder_residual_transformer_gb300 import synth


def test_lock_step_pass_is_the_oracle_forward_pass():
    dims = dict(synth.PRESETS["tiny"], n_layers=3, n_standard_layers=1)
    prompt = synth.tokens(20, dims["vocab"])
    variants = {"none": set(), "all": set(RA.POINTS), **{p: {p} for p in RA.POINTS}}
    res, logits = RA.attribution(dims, prompt, variants, return_logits=True)
    want, _ = O.prefill(dims, O.synthetic_weights(dims), [prompt])
    assert np.array_equal(logits["exact"], want[0])
    assert res["none"] == (0.0, 0.0)
    for p in RA.POINTS:  # 2^-11 relative noise at one point: visible, and far below the logit scale
        assert 0.0 < res[p][0] < 1e-2, p
    assert res["all"][1] > max(res[p][1] for p in RA.POINTS)


def test_fp16_rounding_is_to_nearest_even():
    x = np.array([1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 65504.0, 2.0 ** -24], dtype=np.float32)
    assert RA.fp16(x).tolist() == [1.0, 1.0 + 2.0 ** -9, 65504.0, 2.0 ** -24]
