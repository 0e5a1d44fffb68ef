"""CUDA path vs the CPU oracle, element by element, on the same seeded inputs.

All calls go through the C ABI (libladder.so) via the ctypes binding.
Tolerance on logits: max-abs 3e-2 and relative L2 1e-2 against the fp32
oracle (bf16 weights and KV cache, fp32 accumulation and residual stream).
Integer work (positions, page slots, greedy tokens, lengths) is compared
exactly.
"""
import numpy as np
import pytest
import torch

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import ladder, synth

from gpu_common import (BF16_NAN, check_greedy, compare_logits, gpu_weights, make_model, oracle_weights,
                        packed, prompts_for, small_dims)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    dims = small_dims()
    return dims, gpu_weights(dims), oracle_weights(dims)


def run_teacher_forced(model, prompts, feed, graph=False, standard=None, parallel=None):
    """Prefill then decode feeding feed[:, s]; returns logits [S+1, B, V] and greedy tokens."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        model.set_mode(graph=graph, standard=getattr(model, "_standard", False) if standard is None else standard,
                       parallel=getattr(model, "_parallel", False) if parallel is None else parallel,
                       fast_prefill=getattr(model, "_fast_prefill", False))
        logits, nxt = model.prefill(packed(prompts), [len(p) for p in prompts])
        out, toks = [logits.cpu().numpy()], [nxt.cpu().numpy()]
        tok_dev = torch.empty(len(prompts), dtype=torch.int32, device="cuda")
        lg = torch.empty(len(prompts), model.dims["vocab"], dtype=torch.float32, device="cuda")
        nt = torch.empty(len(prompts), dtype=torch.int32, device="cuda")
        for i in range(feed.shape[1]):
            tok_dev.copy_(torch.from_numpy(feed[:, i].astype(np.int32)))
            model.decode_step(tok_dev, lg, nt)
            out.append(lg.cpu().numpy())
            toks.append(nt.cpu().numpy())
    s.synchronize()
    return np.stack(out), np.stack(toks)


def test_tiny_greedy_tokens_and_logits(tiny):
    dims, gw, ow = tiny
    prompts = prompts_for([16], dims["vocab"])
    o_toks, o_logits, _ = O.greedy_generate(dims, ow, prompts, 8)
    model = make_model(dims, gw, max_batch=1, max_seq=64)
    g_logits, g_toks = run_teacher_forced(model, prompts, o_toks[:, :8])
    errs = [compare_logits(g_logits[s], o_logits[s], f"step {s}")[0] for s in range(9)]
    ties = check_greedy(g_toks[:, 0], o_logits[:, 0], 2 * max(errs))
    print("steps decided by the near-tie rule:", ties)
    # free-running greedy generation on the device (token fed back without the host)
    model.reset()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _, nxt = model.prefill(packed(prompts), [16])
        gen = [nxt.clone()]
        for _ in range(8):
            model.decode_step(nxt, next_tok=nxt)
            gen.append(nxt.clone())
    s.synchronize()
    gen = torch.stack(gen).cpu().numpy()[:, 0]
    srt = np.sort(o_logits[:, 0], axis=-1)
    print("oracle top-2 margins", (srt[:, -1] - srt[:, -2]).round(6).tolist(), "max err", max(errs))
    for s_, (a, b) in enumerate(zip(gen, o_toks[0])):
        if a != b:  # only a near-tie may make the free run diverge, and then the rest follows a new prefix
            check_greedy([a], [o_logits[s_, 0]], 2 * max(errs))
            break


def test_bf16_weights_and_operands():
    """The bf16 storage variant of the prefill kernels and the B <= 2 decode
    kernels against the oracle (the batched projections: the next test)."""
    dims = small_dims()
    ow = oracle_weights(dims)
    lens = [16, 70]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gpu_weights(dims, dtype="bf16"), max_batch=2, max_seq=96, page_size=32)
    g_logits, g_toks = run_teacher_forced(model, prompts, feed, graph=True)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(4):
        compare_logits(g_logits[s_], o_logits[s_], f"bf16 step {s_}")


def test_bf16_batched_decode_on_tensor_cores():
    """bf16 storage on the batched (mma.sync, split-K) decode projections: five
    ragged sequences, prefill and three decode steps."""
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072, vocab=2048,
                      n_layers=2, n_standard_layers=0)
    ow = oracle_weights(dims)
    lens = [9, 40, 23, 3, 61]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(5)])
    model = make_model(dims, gpu_weights(dims, dtype="bf16"), max_batch=5, max_seq=96, page_size=32)
    g_logits, _ = run_teacher_forced(model, prompts, feed, graph=True)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(4):
        compare_logits(g_logits[s_], o_logits[s_], f"bf16 batched step {s_}")


@pytest.mark.parametrize("graph", [False, True])
def test_medium_head_dim_128_and_split_k(graph):
    """head_dim 128 in both attention kernels; at 3 rows the projections take the split-K
    tensor-core path (the down projection's K = 3072 in three slices)."""
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072, vocab=2048,
                      n_layers=2, n_standard_layers=0)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    lens = [100, 257, 3]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(3)])
    model = make_model(dims, gw, max_batch=3, max_seq=320, page_size=64)
    g_logits, _ = run_teacher_forced(model, prompts, feed, graph=graph)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(4):
        compare_logits(g_logits[s_], o_logits[s_], f"medium step {s_}")


@pytest.mark.parametrize("B", [1, 2])
def test_decode_rows_longer_than_one_staged_chunk(B):
    """Decode projections whose rows exceed the GEMV's staging buffer (ffn 20480 > 16384
    columns per batch row): the down projection stages its rows in chunks and splits K
    across warps within each chunk (B = 1: 2 chunks of 10240, K split 4; B = 2: 4 chunks
    of 5120, the launch shapes that fit one wave)."""
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=20480, vocab=2048,
                      n_layers=2, n_standard_layers=0)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    lens = [37, 5][:B]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(B)])
    model = make_model(dims, gw, max_batch=B, max_seq=64, page_size=32)
    g_logits, _ = run_teacher_forced(model, prompts, feed, graph=True)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(4):
        compare_logits(g_logits[s_], o_logits[s_], f"long rows B={B} step {s_}")


def test_kv_cache_layout_is_bit_exact(tiny):
    dims, gw, ow = tiny
    page = 16
    rng = np.random.default_rng(11)
    model = make_model(dims, gw, max_batch=2, max_seq=64, page_size=page, kv_fill_bits=BF16_NAN,
                       page_order=rng.permutation(2 * 4))
    prompts = prompts_for([21, 9], dims["vocab"])
    feed = np.stack([synth.tokens(5, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    run_teacher_forced(model, prompts, feed)
    assert [model.seq_len(0), model.seq_len(1)] == [26, 14]
    assert model.seq_lens.cpu().tolist()[:2] == [26, 14]
    _, caches = O.teacher_forced_decode(dims, ow, prompts, feed)
    pool = model.kv_view().float().cpu().numpy()
    bits = model.kv_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    written = np.zeros(bits.shape, dtype=bool)
    for b, cache in enumerate(caches):
        for p in range(cache.length):
            pg, off = O.kv_slot(model.host_table[b], p, page)
            for l in range(dims["n_layers"]):
                for kv, ref in ((0, cache.k[l]), (1, cache.v[l])):
                    got = pool[l, pg, kv, :, off, :]
                    want = ref[p]
                    assert np.abs(got - want).max() <= 1e-2 * np.abs(want).max() + 1e-3, (b, p, l, kv)
                    for h in range(dims["n_kv_heads"]):
                        o = O.kv_pool_offset(dims["n_kv_heads"], dims["head_dim"], model.num_pages, page,
                                             l, pg, kv, h, off)
                        written[o:o + dims["head_dim"]] = True
    # every slot the oracle does not fill still holds the poison bits, untouched
    assert (bits[~written] == BF16_NAN).all()
    assert not (bits[written] == BF16_NAN).any()


def test_paired_gemm_tiles_in_prefill():
    """4096 packed prompt rows make every prefill projection use 256 x 256 tiles
    computed by CTA pairs (the paired tcgen05 MMA): QKV with RoPE and the K/V
    scatter, gate/up with SwiGLU, and both residual GEMMs."""
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=2048, vocab=2048,
                      n_layers=2, n_standard_layers=0)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    lens = [2048, 2048]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(1, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gw, max_batch=2, max_seq=2112, page_size=64)
    g_logits, _ = run_teacher_forced(model, prompts, feed)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(2):
        compare_logits(g_logits[s_], o_logits[s_], f"paired tiles step {s_}")


def test_narrow_gemm_tiles_with_ragged_rows():
    """450 packed rows (4 m tiles, the last one ragged) with narrow projections
    (N = 768 and 512): QKV and both residual GEMMs take 128-wide tiles with
    two-chunk boxes, the gate/up GEMM 256 x 256 tiles on CTA pairs."""
    dims = small_dims(d_model=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1024, vocab=2048,
                      n_layers=2, n_standard_layers=0)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    lens = [300, 150]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(1, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gw, max_batch=2, max_seq=320, page_size=64)
    g_logits, _ = run_teacher_forced(model, prompts, feed)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(2):
        compare_logits(g_logits[s_], o_logits[s_], f"paired narrow tiles step {s_}")


def test_prefill_repeats_bitwise():
    """500 packed rows (4 m tiles) and d = 1024 (narrow residual GEMMs, paired
    gate/up tiles, two-stream-free prefill with programmatic dependent launch):
    logits match the oracle, and repeated prefills give identical bits."""
    dims = small_dims(d_model=1024, n_q_heads=16, n_kv_heads=4, head_dim=64, ffn_dim=4096, vocab=2048,
                      n_layers=2, n_standard_layers=0)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    lens = [300, 200]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(1, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gw, max_batch=2, max_seq=320, page_size=64)
    g_logits, _ = run_teacher_forced(model, prompts, feed)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(2):
        compare_logits(g_logits[s_], o_logits[s_], f"4-tile prefill step {s_}")
    runs = []
    for _ in range(3):
        model.reset()
        runs.append(run_teacher_forced(model, prompts, feed)[0])
    for r in runs:
        assert np.array_equal(r, g_logits)


FAST_GEOMETRIES = {
    # name: (dims overrides, prompt lengths, weight dtype)
    "narrow ragged": (dict(d_model=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=1024), [300, 150], "fp16"),
    "paired 256x256": (dict(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=2048), [2048, 2048],
                       "fp16"),
    "hd128 split K": (dict(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072), [100, 257, 3],
                      "fp16"),
    "bf16": (dict(), [16, 70], "bf16"),
}


@pytest.mark.parametrize("name", sorted(FAST_GEOMETRIES))
def test_prefill_precisions_match_oracle(name):
    """Both prefill precisions on every GEMM tile shape (128-wide tiles with a
    ragged last m tile, paired 256 x 256 tiles, 256-wide tiles with K in two
    chunks) and on bf16 storage: each within the logit tolerance, the hi/lo
    default strictly closer to the oracle than the once-rounded fast mode, and
    the two not bitwise equal (the lo planes take part)."""
    over, lens, dtype = FAST_GEOMETRIES[name]
    dims = small_dims(vocab=2048, n_layers=2, n_standard_layers=0, **over)
    ow = oracle_weights(dims)
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(2, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(len(lens))])
    model = make_model(dims, gpu_weights(dims, dtype=dtype), max_batch=len(lens), max_seq=max(lens) + 64,
                       page_size=64 if max(lens) > 64 else 32)
    got = {}
    for fast in (False, True):
        model._fast_prefill = fast
        model.reset()
        got[fast] = run_teacher_forced(model, prompts, feed, graph=True)[0]
    model.close()
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    err = {}  # relative L2 error summed over the three steps
    for fast in (False, True):
        err[fast] = sum(compare_logits(got[fast][s], o_logits[s], f"{name} fast={fast} step {s}")[1] for s in range(3))
    print(f"{name}: summed rel-L2 hi/lo {err[False]:.3e}, fast {err[True]:.3e}")
    assert not np.array_equal(got[False], got[True])
    assert err[False] < err[True]


@pytest.mark.parametrize("B", [3, 4, 16, 21])
def test_batched_decode_on_tensor_cores(B):
    """Decode batches of 3 rows and more run on the mma.sync projection in chunks
    of 16 rows (21 = 16 + 5); the down projection (K = 3072) stages its input in
    two chunks, the QKV projection writes rotated K/V for every row."""
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072, vocab=2048,
                      n_layers=2, n_standard_layers=0)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    lens = [(7 * b) % 61 + 3 for b in range(B)]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(B)])
    model = make_model(dims, gw, max_batch=B, max_seq=96, page_size=32)
    g_logits, g_toks = run_teacher_forced(model, prompts, feed, graph=True)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(4):
        compare_logits(g_logits[s_], o_logits[s_], f"B={B} step {s_}")
    # greedy tokens agree unless the oracle's top-2 margin is within twice the logit tolerance
    for s_ in range(4):
        check_greedy(g_toks[s_], o_logits[s_], 6e-2)


def test_maximum_batch_and_full_capacity():
    """The largest batch the library takes (64 sequences: four 16-row chunks of
    the batched projection, 64 prefill segments of ragged lengths from 1 to 126),
    decode to the last position each sequence's pages hold, against the oracle;
    one step more is refused before any launch."""
    dims = small_dims()
    B, cap = 64, 128
    lens = [1 + (37 * b) % 126 for b in range(B)]  # at most cap - 2, so two decode steps fit
    lens[0], lens[1] = cap - 2, 1  # one sequence ends exactly at its capacity
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(2, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(B)])
    model = make_model(dims, gpu_weights(dims), max_batch=B, max_seq=cap, page_size=32,
                       max_prefill_tokens=sum(lens))
    g_logits, _ = run_teacher_forced(model, prompts, feed, graph=True)
    o_logits, _ = O.teacher_forced_decode(dims, oracle_weights(dims), prompts, feed)
    for s_ in range(3):
        compare_logits(g_logits[s_], o_logits[s_], f"B=64 step {s_}")
    assert model.seq_len(0) == cap
    with pytest.raises(ladder.LadderError) as e:
        model.decode_step(torch.zeros(B, dtype=torch.int32, device="cuda"))
    assert e.value.code == ladder.LADDER_ERR_CAPACITY
    model.close()


def test_ragged_batch_prefill_and_decode(tiny):
    dims, gw, ow = tiny
    lens = [5, 70, 33, 1, 64, 17]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(len(lens))])
    model = make_model(dims, gw, max_batch=6, max_seq=96, page_size=32)
    g_logits, g_toks = run_teacher_forced(model, prompts, feed)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    errs = [compare_logits(g_logits[s], o_logits[s], f"step {s}")[0] for s in range(4)]
    # every row of every step: the oracle's argmax unless its top-2 margin is
    # inside twice the observed logit error (then a near-maximal candidate)
    for s in range(4):
        check_greedy(g_toks[s], o_logits[s], 2 * max(errs))


@pytest.mark.parametrize("nstd,strict", [(1, 0), (1, 1), (3, 0)])
def test_hybrid_and_standard_layers(nstd, strict):
    dims = small_dims(n_layers=3, n_standard_layers=nstd)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    prompts = prompts_for([12, 7], dims["vocab"])
    feed = np.stack([synth.tokens(2, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gw, max_batch=2, max_seq=32, page_size=16, strict_boundary=strict)
    g_logits, _ = run_teacher_forced(model, prompts, feed)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed, strict_boundary=bool(strict))
    for s in range(3):
        compare_logits(g_logits[s], o_logits[s], f"nstd {nstd} strict {strict} step {s}")


def test_standard_mode_switch_matches_standard_oracle(tiny):
    dims, gw, _ = tiny
    prompts = prompts_for([16], dims["vocab"])
    feed = synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED)[None, :]
    model = make_model(dims, gw, max_batch=1, max_seq=32)
    model.set_mode(standard=True)
    s = torch.cuda.Stream()
    std_dims = dict(dims, n_standard_layers=dims["n_layers"])
    o_logits, _ = O.teacher_forced_decode(std_dims, oracle_weights(std_dims), prompts, feed)
    with torch.cuda.stream(s):
        model.set_mode(standard=True)
        lg, _ = model.prefill(packed(prompts), [16])
        got = [lg.cpu().numpy()]
        for i in range(3):
            lg, _ = model.decode_step(torch.tensor(feed[:, i], dtype=torch.int32, device="cuda"))
            got.append(lg.cpu().numpy())
    for i in range(4):
        compare_logits(got[i], o_logits[i], f"standard step {i}")
    lad = O.teacher_forced_decode(dims, oracle_weights(dims), prompts, feed)[0]
    assert np.abs(lad - o_logits).max() > 1e-3  # the two schedules really differ


@pytest.mark.parametrize("graph", [False, True])
def test_parallel_mode_matches_parallel_oracle(graph):
    """Every layer a parallel block (both modules read the layer input), on a
    hybrid-configured model: the mode overrides the configured schedule.  Two
    ragged sequences, prefill and four decode steps, eager and graph replay."""
    dims = small_dims(n_layers=3, n_standard_layers=1)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    prompts = prompts_for([37, 12], dims["vocab"])
    feed = np.stack([synth.tokens(4, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gw, max_batch=2, max_seq=64, page_size=16)
    g_logits, g_toks = run_teacher_forced(model, prompts, feed, graph=graph, parallel=True)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed, parallel=True)
    errs = [compare_logits(g_logits[s_], o_logits[s_], f"parallel step {s_}")[0] for s_ in range(5)]
    for s_ in range(5):
        check_greedy(g_toks[s_], o_logits[s_], 2 * max(errs))
    lad = O.teacher_forced_decode(dims, ow, prompts, feed)[0]
    assert np.abs(lad - o_logits).max() > 1e-3  # the schedules really differ


def test_zero_wo_makes_parallel_equal_standard_bitwise():
    """With W_o = 0 the attention adds nothing, so the MLP's input x_{2l} equals
    x_{2l+1}: the parallel and standard schedules give the same bits."""
    dims = small_dims()
    model = make_model(dims, gpu_weights(dims, transform=_bits), max_batch=1, max_seq=32)
    prompts = prompts_for([16], dims["vocab"])
    outs = []
    for parallel in (False, True):
        model.reset()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            model.set_mode(standard=not parallel, parallel=parallel)
            lg, nt = model.prefill(packed(prompts), [16])
            l2, _ = model.decode_step(nt)
        s.synchronize()
        outs.append((lg.cpu().numpy(), l2.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_shard_mode_parallel_schedule():
    """Shard mode (k = 2 row/column shards, reduce on the second stream) with
    parallel blocks."""
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072, vocab=2048)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    prompts = prompts_for([40, 9], dims["vocab"])
    feed = np.stack([synth.tokens(4, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gw, max_batch=2, max_seq=64, page_size=32, shard_k=2)
    g_logits, _ = run_teacher_forced(model, prompts, feed, graph=True, parallel=True)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed, parallel=True)
    for s_ in range(5):
        compare_logits(g_logits[s_], o_logits[s_], f"shard parallel step {s_}")


def _bits(name, layer, b):
    return np.zeros_like(b) if name == "wo" else b


def test_zero_wo_makes_ladder_equal_standard_bitwise():
    dims = small_dims()
    model = make_model(dims, gpu_weights(dims, transform=_bits), max_batch=1, max_seq=32)
    prompts = prompts_for([16], dims["vocab"])
    outs = []
    for standard in (False, True):
        model.reset()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            model.set_mode(standard=standard)
            lg, nt = model.prefill(packed(prompts), [16])
            l2, _ = model.decode_step(nt)
        s.synchronize()
        outs.append((lg.cpu().numpy(), l2.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_graph_replay_equals_eager_and_runs_are_deterministic(tiny):
    dims, gw, _ = tiny
    prompts = prompts_for([16, 40], dims["vocab"])
    feed = np.stack([synth.tokens(6, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    results = []
    for graph, order in ((False, None), (True, None), (False, np.random.default_rng(3).permutation(2 * 2))):
        model = make_model(dims, gw, max_batch=2, max_seq=64, page_size=32, page_order=order)
        results.append(run_teacher_forced(model, prompts, feed, graph=graph))
        model.close()
    for r in results[1:]:
        assert np.array_equal(r[0], results[0][0]) and np.array_equal(r[1], results[0][1])


def test_host_and_device_errors(tiny):
    dims, gw, _ = tiny
    model = make_model(dims, gw, max_batch=2, max_seq=32, page_size=16)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        # a token id outside the vocabulary is reported by the device error word
        bad = torch.tensor([3, dims["vocab"] + 5], dtype=torch.int32, device="cuda")
        model.prefill(bad, [1, 1])
        assert model.device_error(s) == 1
        assert model.device_error(s) == 0
        # prefill on a non-empty sequence and lengths beyond capacity fail before any launch
        with pytest.raises(ladder.LadderError) as e:
            model.prefill(packed(prompts_for([4], dims["vocab"])), [4])
        assert e.value.code == ladder.LADDER_ERR_INVALID
        model.reset()
        with pytest.raises(ladder.LadderError) as e:
            model.prefill(packed(prompts_for([33], dims["vocab"])), [33])
        assert e.value.code == ladder.LADDER_ERR_CAPACITY
        model.prefill(packed(prompts_for([31], dims["vocab"])), [31])
        tok = torch.tensor([1], dtype=torch.int32, device="cuda")
        model.decode_step(tok)
        assert model.seq_len(0) == 32
        with pytest.raises(ladder.LadderError) as e:
            model.decode_step(tok)
        assert e.value.code == ladder.LADDER_ERR_CAPACITY
        assert model.seq_len(0) == 32
        with pytest.raises(ladder.LadderError):
            model.decode_step(torch.zeros(3, dtype=torch.int32, device="cuda"))
        # empty batches and empty prompts are rejected and leave the cache as it was
        for call in (lambda: model.decode_step(torch.zeros(0, dtype=torch.int32, device="cuda")),
                     lambda: model.prefill(torch.zeros(0, dtype=torch.int32, device="cuda"), [])):
            with pytest.raises(ladder.LadderError) as e:
                call()
            assert e.value.code == ladder.LADDER_ERR_INVALID
        model.reset()
        with pytest.raises(ladder.LadderError) as e:
            model.prefill(packed(prompts_for([4], dims["vocab"])), [4, 0])
        assert e.value.code == ladder.LADDER_ERR_INVALID
        assert model.seq_len(0) == 0 and model.seq_len(1) == 0
        model.prefill(packed(prompts_for([31], dims["vocab"])), [31])
        model.decode_step(tok)
    s.synchronize()
    assert model.seq_lens.cpu().tolist()[0] == 32


def test_non_finite_projection_output_is_flagged():
    """A prefill whose SwiGLU activations leave the fp16 range (gate and up
    weights of layer 0 scaled by 2^14, still finite fp16 weights) reports bit 4
    of the device error word; the same model with bf16 storage (no overflow)
    reports nothing."""
    dims = small_dims()

    def scale(name, layer, bits):
        if layer != 0 or name not in ("w_gate", "w_up"):
            return bits
        f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** 14)  # exact: a power of two
        return (f.view(np.uint32) >> 16).astype(np.uint16)

    prompts = prompts_for([24], dims["vocab"])
    codes = {}
    for dtype in ("fp16", "bf16"):
        model = make_model(dims, gpu_weights(dims, transform=scale, dtype=dtype), max_batch=1, max_seq=32,
                           page_size=16)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            model.prefill(packed(prompts), [24])
            codes[dtype] = model.device_error(s)
        model.close()
    assert codes["fp16"] & 4, codes
    assert codes["bf16"] == 0, codes


def test_non_finite_decode_kv_write_is_flagged():
    """A decode step whose new K values leave the fp16 range (the K projection of
    layer 0 scaled by 2^18, still finite fp16 weights) reports bit 4 of the device
    error word from the decode projection's cache write (the prefill's own flags
    are read, and so cleared, first); the same model with bf16 storage reports
    nothing."""
    dims = small_dims()

    def scale(name, layer, bits):
        if layer != 0 or name != "wk":
            return bits
        f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** 18)  # exact: a power of two
        return (f.view(np.uint32) >> 16).astype(np.uint16)

    prompts = prompts_for([24], dims["vocab"])
    codes = {}
    for dtype in ("fp16", "bf16"):
        model = make_model(dims, gpu_weights(dims, transform=scale, dtype=dtype), max_batch=1, max_seq=32,
                           page_size=16)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            _, nt = model.prefill(packed(prompts), [24])
            model.device_error(s)
            model.decode_step(nt)
            codes[dtype] = model.device_error(s)
        model.close()
    assert codes["fp16"] & 4, codes
    assert codes["bf16"] == 0, codes


@pytest.mark.slow
def test_full_size_1p2b_prefill_and_decode():
    """The 1.2B workload at its full prompt length, in the graph-replay launch
    configuration the benchmark times, against the oracle on the same inputs,
    with the prefill GEMM activations as hi/lo pairs (the default) and rounded
    once (fast prefill): both within the logit tolerance at this depth."""
    dims = dict(synth.PRESETS["1.2b"])
    gw = gpu_weights(dims)
    prompts = prompts_for([1024], dims["vocab"])
    feed = synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED)[None, :]
    model = make_model(dims, gw, max_batch=1, max_seq=1024 + 256, max_prefill_tokens=1024)
    runs = {}
    for fast in (False, True):
        model._fast_prefill = fast
        model.reset()
        runs[fast] = run_teacher_forced(model, prompts, feed, graph=True)
    model.close()
    del gw, model
    torch.cuda.empty_cache()
    o_logits, _ = O.teacher_forced_decode(dims, O.synthetic_weights(dims), prompts, feed)
    rel = {}
    for fast, (g_logits, g_toks) in runs.items():
        er = [compare_logits(g_logits[s], o_logits[s], f"1.2B fast={fast} step {s}") for s in range(4)]
        ties = check_greedy(g_toks[:, 0], o_logits[:, 0], 2 * max(e for e, _ in er))
        rel[fast] = sum(r for _, r in er)
        print(f"1.2B fast_prefill={fast}: max-abs {max(e for e, _ in er):.3e} rel-L2 {max(r for _, r in er):.3e}; "
              f"steps decided by the near-tie rule: {ties}")
    assert rel[False] < rel[True]  # the hi/lo operands are the more accurate prefill


@pytest.mark.slow
def test_full_size_1p2b_bf16_storage():
    """The 1.2B workload with bf16 storage (weights, KV cache and the prefill's
    hi/lo tensor-core operands in bf16), the configuration of the bench's bf16
    arm: its full prompt and three decode steps in the graph configuration,
    against the oracle on the same bf16-valued weights."""
    dims = dict(synth.PRESETS["1.2b"])
    prompts = prompts_for([1024], dims["vocab"])
    feed = synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED)[None, :]
    model = make_model(dims, gpu_weights(dims, dtype="bf16"), max_batch=1, max_seq=1024 + 256,
                       max_prefill_tokens=1024)
    g_logits, g_toks = run_teacher_forced(model, prompts, feed, graph=True)
    model.close()
    del model
    torch.cuda.empty_cache()
    o_logits, _ = O.teacher_forced_decode(dims, O.synthetic_weights(dims), prompts, feed)
    er = [compare_logits(g_logits[s], o_logits[s], f"1.2B bf16 step {s}") for s in range(4)]
    ties = check_greedy(g_toks[:, 0], o_logits[:, 0], 2 * max(e for e, _ in er))
    print(f"1.2B bf16 storage: max-abs {max(e for e, _ in er):.3e} rel-L2 {max(r for _, r in er):.3e}; "
          f"steps decided by the near-tie rule: {ties}")


@pytest.mark.parametrize("k,standard,graph", [(2, False, False), (2, True, True), (4, False, True), (4, True, False)])
def test_shard_mode_matches_oracle(k, standard, graph):
    """Shard mode: row-parallel partial sums reduced on a second stream (ladder or standard schedule)."""
    if k == 2:
        dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072, vocab=2048)
    else:
        dims = small_dims(d_model=1024, n_q_heads=16, n_kv_heads=4, head_dim=64, ffn_dim=4096, vocab=2048)
    gw = gpu_weights(dims)
    odims = dict(dims, n_standard_layers=dims["n_layers"]) if standard else dims
    ow = oracle_weights(odims)
    lens = [40, 9]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(4, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gw, max_batch=2, max_seq=64, page_size=32, shard_k=k)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        model.set_mode(standard=standard, graph=graph)
    g_logits, _ = run_teacher_forced(model, prompts, feed, graph=graph)
    o_logits, _ = O.teacher_forced_decode(odims, ow, prompts, feed)
    for s_ in range(5):
        compare_logits(g_logits[s_], o_logits[s_], f"shard k={k} standard={standard} step {s_}")


@pytest.mark.parametrize("k,ffn,B", [(2, 10240, 2), (4, 4096, 4)])
def test_shard_mode_batches_and_wide_ffn(k, ffn, B):
    """Shard mode with the row-parallel partials of 2 rows over a 10240-wide ffn
    (each CTA stages one shard's 5120-column slice of a row: the whole rows would
    not fit its staging buffer) and of 4 rows (batch tile 4), ragged prompts."""
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=4, head_dim=128, ffn_dim=ffn, vocab=2048)
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    lens = [40, 9, 23, 1][:B]
    prompts = prompts_for(lens, dims["vocab"])
    feed = np.stack([synth.tokens(4, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(B)])
    model = make_model(dims, gw, max_batch=B, max_seq=64, page_size=32, shard_k=k)
    g_logits, _ = run_teacher_forced(model, prompts, feed, graph=True)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(5):
        compare_logits(g_logits[s_], o_logits[s_], f"shard k={k} ffn={ffn} B={B} step {s_}")


def test_shard_config_is_validated():
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072, vocab=2048)
    gw = gpu_weights(dims)
    for k, code in ((3, ladder.LADDER_ERR_INVALID), (4, ladder.LADDER_ERR_INVALID)):
        with pytest.raises(ladder.LadderError) as e:
            make_model(dims, gw, max_batch=1, max_seq=32, shard_k=k)
        assert e.value.code == code


@pytest.mark.parametrize("shard_k", [1, 2])
def test_launch_timeline(shard_k):
    """The launch timeline of one eager decode step: every projection,
    attention and reduce launch is recorded once, on the stream the schedule
    puts it on (ladder layers: MLP chain, or shard reduces, on the second
    stream), with end >= start and issue order preserved per stream."""
    dims = small_dims(d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=3072, vocab=2048)
    model = make_model(dims, gpu_weights(dims), max_batch=1, max_seq=64, page_size=32, shard_k=shard_k)
    s = torch.cuda.Stream()
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        model.set_mode(graph=False)
        _, nt = model.prefill(packed(prompts_for([20], dims["vocab"])), [20])
        model.timeline_begin(256, s)
        model.decode_step(nt)
        rows = model.timeline_end()
    s.synchronize()
    L = dims["n_layers"]
    names = [r[1] for r in rows]
    for cls in ("qkv", "attn", "out", "gateup", "down"):
        assert names.count(cls) == L, (cls, names)
    assert names.count("lmhead") == 1
    assert names.count("reduce") == (2 * L if shard_k > 1 else 0)
    for st, cls, t0, t1 in rows:
        assert t1 >= t0 >= 0.0
        if shard_k > 1:
            assert st == (1 if cls == "reduce" else 0), (st, cls)
        elif cls in ("gateup", "down"):
            assert st == 1  # ladder layers: the MLP chain runs on the second stream
        else:
            assert st == 0
    for stream_id in (0, 1):
        starts = [t0 for st, _, t0, _ in rows if st == stream_id]
        assert starts == sorted(starts)


def test_rope_scaling_matches_oracle():
    """Llama-3.1 rotary frequency scaling with the original context set so that
    the tiny model's 32 frequencies fall in all three bands (kept, interpolated,
    divided by the factor); prefill of two ragged prompts and three decode steps."""
    sc = {"factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0, "original_max_position": 64}
    dims = small_dims(rope_scaling=sc)
    f = O.rope_inv_freq(dims["head_dim"], dims["rope_theta"])
    w = 2 * np.pi / f
    assert (w < 16).any() and (w > 64).any() and ((w >= 16) & (w <= 64)).any()
    gw, ow = gpu_weights(dims), oracle_weights(dims)
    prompts = prompts_for([40, 23], dims["vocab"])
    feed = np.stack([synth.tokens(3, dims["vocab"], seed=synth.DECODE_SEED, stream=b) for b in range(2)])
    model = make_model(dims, gw, max_batch=2, max_seq=64, page_size=16)
    g_logits, _ = run_teacher_forced(model, prompts, feed)
    o_logits, _ = O.teacher_forced_decode(dims, ow, prompts, feed)
    for s_ in range(4):
        compare_logits(g_logits[s_], o_logits[s_], f"rope scaling step {s_}")
    plain = O.teacher_forced_decode(dict(dims, rope_scaling=None), ow, prompts, feed)[0]
    assert np.abs(plain - o_logits).max() > 1e-3  # the scaling changes the model
