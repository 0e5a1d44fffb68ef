"""bench.py's multi-rank plumbing on CPU: two gloo ranks, barrier, max of the
timings and sum of the work over ranks (replicas: no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    times = bench.max_over_ranks([1.0 + rank, 10.0 - rank], w)
    work = bench.sum_over_ranks([100.0 * (rank + 1)], w)
    out[rank] = (times, work)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings_and_work():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for rank in range(world):
        times, work = out[rank]
        assert times == [2.0, 10.0]
        assert work == [300.0]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.sum_over_ranks([5.0], 1) == [5.0]


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference times the oracle on the host and prints the
    contract's JSON line; the GPU arm without a GPU fails instead of falling back."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                        "--warmup", "1"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["unit"] == "tok/s" and out["value"] > 0
    assert out["steps"] == 2 and out["warmup"] == 1 and out["higher_is_better"] is True
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["value"] == out["value"]
    assert out["e2e"] == {"value": out["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "fit in L2" in out["config"]["l2"]
    import torch
    if not torch.cuda.is_available():
        r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny", "--steps", "1", "--warmup", "1",
                            "--no-cpu-baseline"], cwd=root, capture_output=True, text=True, timeout=600)
        assert r.returncode != 0 and not r.stdout.strip()


def test_oracle_sample_scales_a_cut_model_by_its_work():
    """The bounded oracle sample of a deep model runs its first layers and
    scales the times by the ratio of algorithmic work; on the full depth the
    scale is 1; the one-thread child process reports the same fields."""
    import bench
    from ladder_residual_transformer_gb300 import synth
    dims = dict(synth.PRESETS["tiny"], n_layers=4)
    cut = bench.sample_dims(dims, 2)
    assert cut["n_layers"] == 2 and cut["n_standard_layers"] == 0
    r = bench.oracle_sample(dims, 8, 2, layers=2)
    assert r["layers"] == 2 and r["decode_tok_s"] > 0 and r["prefill_tok_s"] > 0
    assert bench.decode_step_bytes(dims, [8]) > bench.decode_step_bytes(cut, [8])
    full = bench.oracle_sample(dims, 8, 2)
    assert full["layers"] == 4
    one = bench.one_core_sample("tiny", 8, 2, 2)
    assert one["cores"] == 1 and one["layers"] == 2 and one["value"] > 0
