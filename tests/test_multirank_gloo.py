"""The multi-rank path on CPU ranks (gloo, world size 2): the token
partition covers the batch exactly, per-rank results concatenate to the
single-process result, and the bench's max-over-ranks timing reduction
returns the slowest rank's time on every rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _token_range():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_shard", os.path.join(ROOT, "depth_wise_attention_block_gb300", "shard.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.token_range


def test_token_range_partitions_exactly():
    token_range = _token_range()
    for T in [0, 1, 7, 64, 4096, 4097]:
        for world in [1, 2, 3, 8]:
            spans = [token_range(T, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        token_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    sys.path.insert(0, ROOT)
    import bench
    token_range = _token_range()
    inp = W.block_bf16(T=37, d=64, seed=3, device="cpu")
    t0, t1 = token_range(37, rank, world)
    r, a = O.depth_attention(inp.H[:, t0:t1].double().numpy(), inp.w.double().numpy())
    # gather variable-length shards through fixed-size padded buffers
    pad = 19
    rb = torch.zeros(pad, 64, dtype=torch.float64)
    rb[: t1 - t0] = torch.from_numpy(r)
    gathered = [torch.zeros_like(rb) for _ in range(world)]
    dist.all_gather(gathered, rb)
    slowest = bench.max_over_ranks(1.0 + rank, world, "cpu")
    if rank == 0:
        parts = [g[: token_range(37, k, world)[1] - token_range(37, k, world)[0]] for k, g in enumerate(gathered)]
        queue.put({"r": torch.cat(parts).numpy(), "slowest": slowest})
    else:
        assert slowest == float(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_match_single_process():
    world = 2
    queue = mp.get_context("spawn").SimpleQueue()
    mp.spawn(_worker, args=(world, _free_port(), queue), nprocs=world, join=True)
    res = queue.get()
    inp = W.block_bf16(T=37, d=64, seed=3, device="cpu")
    r_full, _ = O.depth_attention(inp.H.double().numpy(), inp.w.double().numpy())
    assert np.array_equal(res["r"], r_full)
    assert res["slowest"] == float(world)
