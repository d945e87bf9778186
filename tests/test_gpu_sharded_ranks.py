"""The token-sharded multi-rank path through the library, on one GPU.

Two processes (gloo for the gather; each its own CUDA context on cuda:0,
no kernel of one ever waiting on the other) own contiguous token ranges
(shard.token_range) of the K3-width single layer and of a 14-layer stack
(single-pass schedule), run them through the library, and gather the
results.  Tokens are independent and each is computed whole by one CTA in a
fixed order, so the gathered rows equal a single-process run bit for bit.
(The two-phase schedule's tensor-core logits split the channel sum by a
count that follows T, so there sharding changes rounding, not results.)
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
T_LAYER, T_STACK = 1000, 50


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _single_layer(A, H, w):
    S, T, d = H.shape
    r = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    a = torch.empty((T, S), device="cuda")
    A.attnres_aggregate([H[s] for s in range(S)], w, r, a)
    return r, a


def _stack(stk, t0, t1):
    from depth_wise_attention_block_gb300.stack import StackForward
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fwd = StackForward(stk.h0[t0:t1].contiguous(), stk.W, stk.G, stk.Sc, stk.num_layers, stk.block_size,
                       dev_err=err)
    fwd.run()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return fwd.r, torch.cat(fwd.weights, dim=1)


def _bits(r):
    """bf16 rows as int32 bit patterns (gloo carries no 16-bit integers)."""
    return r.view(torch.int16).to(torch.int32)


def _gather(x, t0, t1, T, world):
    """Rows [t0, t1) of every rank into one [T, ...] CPU tensor (padded
    all_gather over gloo)."""
    from depth_wise_attention_block_gb300.shard import token_range
    pad = max(b - a for a, b in (token_range(T, k, world) for k in range(world)))
    buf = torch.zeros((pad,) + tuple(x.shape[1:]), dtype=x.dtype)
    buf[: t1 - t0] = x.cpu()
    parts = [torch.zeros_like(buf) for _ in range(world)]
    dist.all_gather(parts, buf)
    return torch.cat([p[: b - a] for p, (a, b) in zip(parts, (token_range(T, k, world) for k in range(world)))])


def _worker(rank, world, port, out_path):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    import depth_wise_attention_block_gb300 as A
    from depth_wise_attention_block_gb300.shard import token_range
    out = {}
    inp = W.block_bf16(T=T_LAYER, seed=1, device="cuda")          # every rank draws the same batch
    t0, t1 = token_range(T_LAYER, rank, world)
    r, a = _single_layer(A, inp.H[:, t0:t1], inp.w)
    torch.cuda.synchronize()
    out["layer_r"], out["layer_a"] = _gather(_bits(r), t0, t1, T_LAYER, world), _gather(a, t0, t1, T_LAYER, world)
    stk = W.stack(T=T_STACK, num_layers=14, block_size=4, seed=5, device="cuda")
    t0, t1 = token_range(T_STACK, rank, world)
    r, a = _stack(stk, t0, t1)
    torch.cuda.synchronize()
    out["stack_r"], out["stack_a"] = _gather(_bits(r), t0, t1, T_STACK, world), _gather(a, t0, t1, T_STACK, world)
    if rank == 0:
        torch.save(out, out_path)       # a file, not a pipe: the parent reads it after the join
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_on_token_shards_equal_one_process(tmp_path):
    import depth_wise_attention_block_gb300 as A
    world, out_path = 2, str(tmp_path / "rank0.pt")
    mp.spawn(_worker, args=(world, _free_port(), out_path), nprocs=world, join=True)
    got = {k: v.numpy() for k, v in torch.load(out_path).items()}
    inp = W.block_bf16(T=T_LAYER, seed=1, device="cuda")
    r, a = _single_layer(A, inp.H, inp.w)
    stk = W.stack(T=T_STACK, num_layers=14, block_size=4, seed=5, device="cuda")
    sr, sa = _stack(stk, 0, T_STACK)
    torch.cuda.synchronize()
    assert (got["layer_r"] == _bits(r).cpu().numpy()).all()
    assert (got["layer_a"] == a.cpu().numpy()).all()
    assert (got["stack_r"] == _bits(sr).cpu().numpy()).all()
    assert (got["stack_a"] == sa.cpu().numpy()).all()
