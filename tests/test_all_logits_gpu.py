"""Prefill with the logits of every position (LADDER_FLAG_ALL_LOGITS).

Every packed row against the oracle's all-position forward pass, and causality
as a property that holds at any size: changing the token at position p leaves
the logits of positions before p bitwise unchanged (each row of every prefill
kernel depends only on its own inputs and on earlier positions, in a fixed
order), and changes them from p on.
"""
import numpy as np
import pytest
import torch

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import ladder, synth

from gpu_common import compare_logits, gpu_weights, make_model, oracle_weights, packed, prompts_for, small_dims

pytestmark = pytest.mark.gpu


def prefill_all(model, prompts, graph=False):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        model.reset()
        model.set_mode(graph=graph, all_logits=True)
        logits, tok = model.prefill(packed(prompts), [len(p) for p in prompts])
        out = logits.cpu().numpy(), tok.cpu().numpy()
    s.synchronize()
    return out


@pytest.mark.parametrize("max_batch", [3, 2])
def test_every_row_matches_the_oracle(max_batch):
    """Ragged prompts (lm_head over 3 rows per launch: the batched projection
    path; or 2: the per-row one), then a decode step on the filled cache."""
    dims = small_dims()
    lens = [5, 40, 17][:max_batch]
    prompts = prompts_for(lens, dims["vocab"])
    model = make_model(dims, gpu_weights(dims), max_batch=max_batch, max_seq=64, page_size=16)
    g_all, g_tok = prefill_all(model, prompts)
    assert g_all.shape == (sum(lens), dims["vocab"])
    o_all = O.forward(dims, oracle_weights(dims), prompts, [O.SeqCache() for _ in lens], all_positions=True)
    r = 0
    for b, n in enumerate(lens):
        compare_logits(g_all[r:r + n], o_all[b], f"sequence {b}")
        assert g_tok[b] == O.argmax_lowest(g_all[r + n - 1])  # the device's own last row
        r += n
    # the cache is filled as in the ordinary prefill: one decode step matches the oracle
    feed = np.array([7, 300, 11][:max_batch], dtype=np.int32)
    lg, _ = model.decode_step(torch.from_numpy(feed).cuda())
    caches = O.prefill(dims, oracle_weights(dims), prompts)[1]
    compare_logits(lg.cpu().numpy(), O.decode_step(dims, oracle_weights(dims), feed, caches), "decode after all-row prefill")


def test_flag_checks():
    dims = small_dims()
    model = make_model(dims, gpu_weights(dims), max_batch=2, max_seq=32, page_size=16)
    model.set_sampling(0.8, 5, 1)
    model.set_mode(all_logits=True)
    with pytest.raises(ladder.LadderError) as e:
        model.prefill(packed(prompts_for([4], dims["vocab"])), [4])
    assert e.value.code == ladder.LADDER_ERR_UNSUPPORTED
    assert model.seq_len(0) == 0
    # without a next-token output (NULL), sampling settings do not matter
    lg = torch.empty(4, dims["vocab"], device="cuda")
    toks = packed(prompts_for([4], dims["vocab"]))
    lens = np.array([4], dtype=np.int32)
    ladder.check(ladder.lib().ladder_prefill(model._m, model._kv, toks.data_ptr(), lens.ctypes.data_as(ladder._pi32),
                                             1, lg.data_ptr(), None, torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert model.seq_len(0) == 4 and np.isfinite(lg.cpu().numpy()).all()
    assert ladder.lib().ladder_set_mode(model._m, 0, 16) == ladder.LADDER_ERR_INVALID


def causality(dims, model, prompt, p):
    a, _ = prefill_all(model, [prompt])
    changed = prompt.copy()
    changed[p] = (changed[p] + 1) % dims["vocab"]
    b, _ = prefill_all(model, [changed])
    assert np.array_equal(a[:p], b[:p]), "rows before the changed token moved"
    assert not np.array_equal(a[p], b[p])
    return a


def test_causality_is_bitwise_tiny():
    dims = small_dims()
    model = make_model(dims, gpu_weights(dims), max_batch=1, max_seq=160, page_size=32)
    prompt = prompts_for([150], dims["vocab"])[0]
    for p in (0, 63, 128, 149):
        causality(dims, model, prompt, p)


@pytest.mark.slow
def test_full_size_1p2b_every_row_and_causality():
    """The 1.2B workload's 1024-token prompt: every row against the oracle, and
    causality at position 700."""
    dims = dict(synth.PRESETS["1.2b"])
    gw = gpu_weights(dims)
    prompt = prompts_for([1024], dims["vocab"])[0]
    model = make_model(dims, gw, max_batch=1, max_seq=1024 + 256, max_prefill_tokens=1024)
    g_all = causality(dims, model, prompt, 700)
    del gw, model
    torch.cuda.empty_cache()
    o_all = O.forward(dims, O.synthetic_weights(dims), [prompt], [O.SeqCache()], all_positions=True)[0]
    for r0 in range(0, 1024, 256):
        compare_logits(g_all[r0:r0 + 256], o_all[r0:r0 + 256], f"1.2B rows {r0}..{r0 + 255}")


# Rows of sequence 0 of the 8B hybrid's 4 x 4096 prefill compared with the oracle:
# the first, a stride of 256 through the sequence, and the last.
SAMPLED_ROWS = [0] + list(range(255, 4096, 256))


@pytest.mark.slow
def test_full_size_8b_hybrid_batch_independence_and_causality():
    """The 8B hybrid's prefill workload (4 x 4096 tokens, the launch shapes the
    benchmark times): a sample of sequence 0's rows (every 256th and the last)
    against the oracle's forward pass of that sequence, and changing one token
    of sequence 2 leaves every row of the other sequences, and the rows of
    sequence 2 before it, bitwise unchanged.  Compared on the device (the
    logits are 8.4 GB).  Then four teacher-forced decode steps of the 4 rows from
    context 4096; sequence 0's logits against the oracle's."""
    dims = dict(synth.PRESETS["8b-hybrid"])
    n, B, p = 4096, 4, 3000
    gw = gpu_weights(dims)
    model = make_model(dims, gw, max_batch=B, max_seq=n + 8, max_prefill_tokens=B * n)
    prompts = prompts_for([n] * B, dims["vocab"])
    feed = np.stack([synth.tokens(4, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(B)])
    seq0 = prompts[0]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        model.set_mode(all_logits=True)
        a, ta = model.prefill(packed(prompts), [n] * B)
        sampled = a[SAMPLED_ROWS].cpu().numpy()
        prompts[2] = prompts[2].copy()
        prompts[2][p] = (prompts[2][p] + 1) % dims["vocab"]
        model.reset()
        b, tb = model.prefill(packed(prompts), [n] * B)
        same_others = all(torch.equal(a[q * n:(q + 1) * n], b[q * n:(q + 1) * n]) for q in (0, 1, 3))
        same_before = torch.equal(a[2 * n:2 * n + p], b[2 * n:2 * n + p])
        moved_at = not torch.equal(a[2 * n + p], b[2 * n + p])
        finite = bool(torch.isfinite(a).all())
        toks = ta.cpu().numpy(), tb.cpu().numpy()
        dec = []
        tok = torch.empty(B, dtype=torch.int32, device="cuda")
        for i in range(feed.shape[1]):
            tok.copy_(torch.from_numpy(feed[:, i].astype(np.int32)))
            lg, _ = model.decode_step(tok)
            dec.append(lg[0].cpu().numpy())
    s.synchronize()
    model.close()
    del a, b, gw, model
    torch.cuda.empty_cache()
    assert finite
    assert same_others, "a sequence's logits depend on another sequence's tokens"
    assert same_before, "rows before the changed token moved"
    assert moved_at
    assert toks[0][[0, 1, 3]].tolist() == toks[1][[0, 1, 3]].tolist()
    # the oracle's stream for sequence 0 alone (sequences are independent, as shown
    # above), extended by its fed tokens: rows n .. n + 3 are the decode steps'
    # logits (cached decode equals re-running the forward pass)
    W = O.synthetic_weights(dims, keep_layers=False)
    rows = SAMPLED_ROWS + [n + i for i in range(feed.shape[1])]
    _, hist = O.forward(dims, W, [np.concatenate([seq0, feed[0]]).astype(np.int32)], [O.SeqCache()],
                        return_stream=True)
    xl = hist[0][2 * dims["n_layers"]][rows]
    del hist
    want = O.rmsnorm(xl, W.glob("final_norm"), dims["norm_eps"]) @ W.glob("lm_head").T
    for i, r in enumerate(SAMPLED_ROWS):
        compare_logits(sampled[i], want[i], f"8B hybrid 4 x 4096 prefill, sequence 0 row {r}")
    for i in range(feed.shape[1]):
        compare_logits(dec[i], want[len(SAMPLED_ROWS) + i], f"8B hybrid, 4 rows from context 4096, decode step {i + 1}")
