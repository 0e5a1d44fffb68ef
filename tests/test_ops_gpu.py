"""Kernel-level parity through the C ABI: standalone decode attention against
the oracle's causal GQA attention on random bf16 caches with permuted pages."""
import math

import numpy as np
import pytest
import torch

import oracle.ladder_oracle as O
from ladder_residual_transformer_gb300 import ladder

pytestmark = pytest.mark.gpu


def to_bf16_bits(a):
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def attention_case(hd, nq, nkv, ps, positions, seed):
    rng = np.random.default_rng(seed)
    B = len(positions)
    max_pos = max(positions)
    pps = (max_pos + 1 + ps - 1) // ps
    num_pages = B * pps
    bits = to_bf16_bits(rng.standard_normal((num_pages, 2, nkv, ps, hd)))
    pool = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    table = rng.permutation(num_pages).astype(np.int32).reshape(B, pps)
    q = rng.standard_normal((B, nq * hd)).astype(np.float32)
    dev = "cuda"
    out = ladder.attention_decode(torch.from_numpy(q).to(dev), torch.from_numpy(bits.view(np.int16)).to(dev),
                                  torch.from_numpy(table).to(dev),
                                  torch.tensor(positions, dtype=torch.int32, device=dev), nkv, hd, ps, max_pos)
    got = out.cpu().numpy().astype(np.float64)
    want = np.empty_like(got)
    for b, p in enumerate(positions):
        slots = [O.kv_slot(table[b], t, ps) for t in range(p + 1)]
        K = np.stack([pool[pg, 0, :, off, :] for pg, off in slots])
        V = np.stack([pool[pg, 1, :, off, :] for pg, off in slots])
        qb = q[b].astype(np.float64).reshape(1, nq, hd)
        want[b] = O.causal_gqa_attention(qb, K, V, np.array([p]), np.arange(p + 1)).reshape(-1)
    return got, want


@pytest.mark.parametrize("hd,nq,nkv,ps", [(64, 32, 8, 64), (128, 64, 8, 16), (64, 4, 4, 32), (128, 8, 1, 64)])
def test_attention_decode_matches_oracle(hd, nq, nkv, ps):
    got, want = attention_case(hd, nq, nkv, ps, [0, 127, 128, 500, 800], seed=hd + nq + ps)
    err = np.abs(got - want).max() / np.abs(want).max()
    assert err < 1e-4, err


def test_attention_decode_rejects_bad_arguments():
    dev = "cuda"
    q = torch.zeros(1, 256, device=dev)
    pool = torch.zeros(4 * 2 * 2 * 64 * 64, dtype=torch.int16, device=dev)
    bt = torch.zeros(1, 4, dtype=torch.int32, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(ladder.LadderError) as e:  # scratch too small
        ladder.attention_decode(q, pool, bt, pos, 2, 64, 64, 200, scratch=torch.empty(16, dtype=torch.uint8, device=dev))
    assert e.value.code == ladder.LADDER_ERR_CAPACITY
    with pytest.raises(ladder.LadderError) as e:  # pages cannot hold max_position
        ladder.attention_decode(q, pool, bt, pos, 2, 64, 64, 300)
    assert e.value.code == ladder.LADDER_ERR_CAPACITY
    with pytest.raises(ladder.LadderError) as e:  # 96 is not a supported head size
        ladder.attention_decode(torch.zeros(1, 192, device=dev), pool, bt, pos, 2, 96, 64, 10)
    assert e.value.code == ladder.LADDER_ERR_UNSUPPORTED
