"""The decode-attention entry point that allocates nothing.

Callers that cannot allocate device memory (work issued while a CUDA graph is
being captured, plugins inside a framework that owns every device buffer,
loops that must not stall on an allocation) use
ladder_attention_decode_noalloc, whose per-split scratch is a static device
array inside the library.  Its results must equal those of
ladder_attention_decode, which takes a caller-provided scratch buffer, call
after call.  This file is collected last so that a failure here leaves every
other test already run.
"""
import numpy as np
import pytest
import torch

from ladder_residual_transformer_gb300 import ladder

pytestmark = pytest.mark.gpu


def make_inputs(seed, B, nq, nkv, hd, ps, positions):
    g = torch.Generator().manual_seed(seed)
    max_pos = max(positions)
    pps = (max_pos + 1 + ps - 1) // ps
    pool = (torch.randn(B * pps, 2, nkv, ps, hd, generator=g) * 0.5).to(torch.bfloat16)
    table = torch.randperm(B * pps, generator=g).to(torch.int32).reshape(B, pps)
    q = torch.randn(B, nq * hd, generator=g)
    dev = "cuda"
    return (q.to(dev), pool.to(dev), table.to(dev), torch.tensor(positions, dtype=torch.int32, device=dev), max_pos)


@pytest.mark.parametrize("shape", [(3, 32, 8, 64, 64, [0, 130, 1000]), (2, 64, 8, 128, 16, [255, 2047])])
def test_noalloc_matches_scratch_entry_point_on_consecutive_calls(shape):
    B, nq, nkv, hd, ps, positions = shape
    for call in range(2):
        q, pool, table, pos, max_pos = make_inputs(100 * call + hd, B, nq, nkv, hd, ps, positions)
        ref = ladder.attention_decode(q, pool, table, pos, nkv, hd, ps, max_pos)
        out = torch.full_like(ref, float("nan"))
        ladder.attention_decode_noalloc(q, pool, table, pos, nkv, hd, ps, max_pos, out)
        torch.cuda.synchronize()
        a, b = out.cpu().numpy(), ref.cpu().numpy()
        assert np.isfinite(a).all()
        assert np.abs(a - b).max() <= 1e-6 * np.abs(b).max(), (call, np.abs(a - b).max())


def test_noalloc_rejects_scratch_beyond_its_static_array():
    # 64 sequences x 64 heads x 64 splits x 130 floats is far above the static array
    dev = "cuda"
    B, nq, nkv, hd, ps, max_pos = 64, 64, 8, 128, 64, 8191
    q = torch.zeros(B, nq * hd, device=dev)
    pool = torch.zeros(1, 2, nkv, ps, hd, dtype=torch.bfloat16, device=dev)
    table = torch.zeros(B, (max_pos + ps) // ps, dtype=torch.int32, device=dev)
    pos = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.empty(B, nq * hd, device=dev)
    with pytest.raises(ladder.LadderError) as e:
        ladder.attention_decode_noalloc(q, pool, table, pos, nkv, hd, ps, max_pos, out)
    assert e.value.code == ladder.LADDER_ERR_CAPACITY
    assert "static array" in str(e.value)
