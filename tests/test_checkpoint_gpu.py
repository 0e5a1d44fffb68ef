"""A Llama-layout checkpoint through the loader and the CUDA path.

The file holds random bf16 tensors under the Hugging Face names, with W_q and
W_k rows in the half-split rotary order.  The loader reorders them for the
library's interleaved pairing; the oracle runs on the file's own tensors with
the half-split pairing.  Hybrid layout (one standard layer under two ladder
layers), Llama-3.1 rotary scaling, two ragged prompts and three decode steps.
"""
import numpy as np
import pytest

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import checkpoint as C
from ladder_residual_transformer_gb300 import ladder, synth

from gpu_common import compare_logits, prompts_for
from test_checkpoint_cpu import SCALING, hf_checkpoint
from test_parity_gpu import run_teacher_forced

pytestmark = pytest.mark.gpu

DIMS = dict(synth.PRESETS["tiny"], n_layers=3, n_standard_layers=1)


@pytest.mark.parametrize("tied,dtype,graph", [(False, "fp16", True), (True, "bf16", False)])
def test_checkpoint_model_matches_the_oracle(tmp_path, tied, dtype, graph):
    bits = hf_checkpoint(tmp_path, DIMS, tied=tied, rope_scaling=SCALING, std=0.02, gain_std=0.1)
    dims, w = C.load_llama(str(tmp_path), n_standard_layers=1, device="cuda", dtype=dtype)
    model = ladder.LadderModel(dims, w, max_batch=2, max_seq=64, page_size=16)
    prompts = prompts_for([13, 30], dims["vocab"])
    feed = np.stack([synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    g_logits, _ = run_teacher_forced(model, prompts, feed, graph=graph)
    ref_dims = dict(dims, rope_interleaved=0)
    W = O.OracleWeights(ref_dims, lambda k, l: synth.bf16_bits_to_f32(bits[C.hf_name(k, l)]))
    o_logits, _ = O.teacher_forced_decode(ref_dims, W, prompts, feed)
    for s in range(4):
        compare_logits(g_logits[s], o_logits[s], f"checkpoint step {s}")
