"""Temperature / top-k sampling on the GPU vs the oracle's sampler.

The sampled token is an argmax of l_i / T - ln(-ln u_i) over the top-k set, so
floating point decides an integer.  Both sides see the same fp32 logits (the
GPU's, downloaded) and the same uniforms u_i (exact in fp32); the kernel scores
in fp32 with CUDA's logf, the oracle in fp64.  So: the top-k set is compared
exactly, the token must be a valid argmax (its oracle score within SCORE_TOL of
the best), and where the oracle's best score leads the runner-up by more than
2 * SCORE_TOL the tokens must be identical.
"""
import numpy as np
import pytest
import torch

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import ladder

from gpu_common import compare_logits, gpu_weights, make_model, oracle_weights, packed, prompts_for, small_dims

pytestmark = pytest.mark.gpu

# fp32 rounding of l * (1/T) (|l/T| <~ 50) and of the two logarithms (|ln(-ln u)| < 17)
SCORE_TOL = 2e-4


def check_sampled(tok, logits_row, T, k, seed, row, pos, what=""):
    l = np.asarray(logits_row, dtype=np.float32).astype(np.float64)
    V = l.shape[0]
    want, score = O.sample_token(l, T, k, seed, row, pos, return_scores=True)
    assert 0 <= tok < V, f"{what}: token {tok} out of range"
    if 0 < k < V:
        pivot = np.sort(l)[V - k]
        assert l[tok] >= pivot, f"{what}: token {tok} outside the top-{k} set"
    best = score[want]
    assert score[tok] >= best - SCORE_TOL * (1 + abs(best)), f"{what}: token {tok} score {score[tok]} vs best {best}"
    s2 = np.sort(score)[-2] if V > 1 else -np.inf
    if best - s2 > 2 * SCORE_TOL * (1 + abs(best)):
        assert tok == want, f"{what}: token {tok} != oracle {want} (margin {best - s2:.3e})"
    return tok == want


@pytest.mark.parametrize("T,k", [(1.0, 0), (0.7, 50), (1.3, 1000), (0.5, 1), (2.0, 128256), (1.0, 300000),
                                 (1e-7, 0)])
def test_sampler_kernel_large_vocab(T, k):
    """128256-entry rows with a spread of logits (a few large ones, many near
    zero), four rows at different positions, through ladder_sample."""
    V, B, seed = 128256, 4, 1234
    rng = np.random.default_rng(17)
    logits = (rng.standard_normal((B, V)) * 2.0).astype(np.float32)
    logits[:, rng.integers(0, V, 40)] += 6.0
    pos = np.array([5, 100, 1023, 7], dtype=np.int32)
    d_logits = torch.from_numpy(logits).cuda()
    d_pos = torch.from_numpy(pos).cuda()
    out = ladder.sample(d_logits, d_pos, T, k, seed, pos_offset=3).cpu().numpy()
    for b in range(B):
        check_sampled(int(out[b]), logits[b], T, k, seed, b, int(pos[b]) + 3, f"T={T} k={k} row {b}")


def test_sampler_ties_at_the_pivot_and_negative_logits():
    """Many logits equal to the k-th largest: all of them stay candidates, and
    over many draws each of them is sampled (the kernel and the oracle agree
    draw by draw)."""
    V, B = 5000, 64
    logits = np.full((B, V), -3.0, dtype=np.float32)
    logits[:, 100:110] = 1.5  # ten-way tie straddling k = 4
    logits[:, 7] = 2.0
    logits[:, 4999] = 2.0
    pos = np.arange(B, dtype=np.int32)
    out = ladder.sample(torch.from_numpy(logits).cuda(), torch.from_numpy(pos).cuda(), 0.9, 4, 99).cpu().numpy()
    agree = sum(check_sampled(int(out[b]), logits[b], 0.9, 4, 99, b, b, f"row {b}") for b in range(B))
    assert agree >= B - 2  # rows whose best two scores tie within the tolerance may differ validly
    assert set(out.tolist()) <= {7, 4999, *range(100, 110)}
    assert len(set(out.tolist()) & set(range(100, 110))) >= 3


def test_sampler_distribution():
    """20000 rows with the same seven logits: frequencies follow softmax(l / T)
    over the top-4 set (chi-square, tail probability ~1e-6)."""
    l = np.array([1.2, -0.3, 0.8, 2.0, 0.0, -1.5, 0.5], dtype=np.float32)
    N, T, k = 20000, 0.8, 4
    logits = np.tile(l, (N, 1))
    pos = np.zeros(N, dtype=np.int32)
    out = ladder.sample(torch.from_numpy(logits).cuda(), torch.from_numpy(pos).cuda(), T, k, 5).cpu().numpy()
    counts = np.bincount(out, minlength=len(l)).astype(np.float64)
    keep = l >= np.sort(l)[len(l) - k]
    p = np.where(keep, np.exp(l / T - (l / T).max()), 0.0)
    p /= p.sum()
    assert np.all(counts[~keep] == 0)
    stat = (((counts - N * p) ** 2 / np.where(p > 0, N * p, 1.0))[keep]).sum()
    assert stat < 30.0, (stat, counts / N, p)


def test_sampler_rejects_bad_arguments():
    d = torch.zeros(2, 10, device="cuda")
    p = torch.zeros(2, dtype=torch.int32, device="cuda")
    for T in (0.0, -1.0, float("nan")):
        with pytest.raises(ladder.LadderError) as e:
            ladder.sample(d, p, T, 0, 0)
        assert e.value.code == ladder.LADDER_ERR_INVALID


@pytest.mark.parametrize("graph", [False, True])
def test_model_sampling_free_running(graph):
    """A model with temperature / top-k sampling: prefill of two ragged prompts,
    then six decode steps fed with the device's own sampled tokens.  Each token
    is checked against the oracle's sampler on the device's logits (positions:
    prompt length, then one more per step), and the logits against the oracle
    run on the same tokens."""
    dims = small_dims()
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    prompts = prompts_for([16, 9], dims["vocab"])
    T, k, seed, steps = 0.8, 20, 11, 6
    model = make_model(dims, gw, max_batch=2, max_seq=64, page_size=16)
    model.set_sampling(T, k, seed)
    s = torch.cuda.Stream()
    logits_all, toks_all = [], []
    with torch.cuda.stream(s):
        model.set_mode(graph=graph)
        lg, nt = model.prefill(packed(prompts), [16, 9])
        logits_all.append(lg.cpu().numpy())
        toks_all.append(nt.cpu().numpy())
        for _ in range(steps):
            lg, nt = model.decode_step(nt)
            logits_all.append(lg.cpu().numpy())
            toks_all.append(nt.cpu().numpy())
    s.synchronize()
    lens = [16, 9]
    for st in range(steps + 1):
        for b in range(2):
            check_sampled(int(toks_all[st][b]), logits_all[st][b], T, k, seed, b, lens[b] + st, f"step {st} row {b}")
    feed = np.stack(toks_all[:steps], axis=1)  # token fed at step s = sampled at step s - 1
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for st in range(steps + 1):
        compare_logits(logits_all[st], o_logits[st], f"sampled run step {st}")
    # switching back to greedy: the prefill token is the argmax of the same logits
    model.set_sampling(0.0)
    model.reset()
    with torch.cuda.stream(s):
        _, g0 = model.prefill(packed(prompts), [16, 9])
    s.synchronize()
    assert np.array_equal(g0.cpu().numpy(), O.argmax_lowest(logits_all[0]))
