"""Writes tests/golden/tiny_greedy.json from the CPU oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
The file is a regression record of the oracle on the tiny workload (2 ladder
layers, d_model 256, 16-token prompt from seed 1, weights from seed 0, 8 greedy
steps): the 9 greedy tokens, the first 8 logits of each step, and the top-2
margin of each step.  It calls nothing but oracle/ and the seeded generator.
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle.ladder_oracle as O  # noqa: E402
from ladder_residual_transformer_gb300 import synth  # noqa: E402

dims = dict(synth.PRESETS["tiny"])
toks, logits, _ = O.greedy_generate(dims, O.synthetic_weights(dims), [synth.tokens(16, dims["vocab"])], 8)
srt = np.sort(logits[:, 0, :], axis=-1)
out = {
    "workload": "tiny: 2 ladder layers, d_model 256, 4 q / 2 kv heads, hd 64, ffn 768, vocab 1024; prompt 16 tokens (seed 1), weights seed 0; 8 greedy steps",
    "tokens": toks[0].tolist(),
    "logits_head": logits[:, 0, :8].astype(float).round(7).tolist(),
    "top2_margin": (srt[:, -1] - srt[:, -2]).astype(float).tolist(),
}
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_greedy.json"), "w") as f:
    json.dump(out, f, indent=1)
print(out["tokens"], out["top2_margin"])
