"""Pipeline-parallel transfer plan (depth_wise_attention_block_gb300/pipeline.py):
host logic checked on CPU, and a two-rank gloo pipeline that runs a 93-layer
stack split across ranks, exchanging only the planned buffers, and must
reproduce the single-process oracle exactly."""
import importlib.util
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pipeline():
    """pipeline.py by path (host logic: no need for the CUDA library here)."""
    import sys
    if "_attnres_pipeline" not in sys.modules:
        spec = importlib.util.spec_from_file_location(
            "_attnres_pipeline", os.path.join(ROOT, "depth_wise_attention_block_gb300", "pipeline.py"))
        mod = importlib.util.module_from_spec(spec)
        sys.modules["_attnres_pipeline"] = mod
        spec.loader.exec_module(mod)
    return sys.modules["_attnres_pipeline"]


CONTIGUOUS = [(0, 1, 47), (1, 48, 93)]                       # boundary inside block 4 (37..48)
INTERLEAVED = [(0, 1, 20), (1, 21, 45), (0, 46, 70), (1, 71, 93)]


@pytest.mark.parametrize("chunks", [CONTIGUOUS, INTERLEAVED, [(0, 1, 36), (1, 37, 93)],
                                    [(0, 1, 10), (1, 11, 30), (2, 31, 60), (3, 61, 93)]])
def test_plan_gives_each_chunk_its_eq10_sources(chunks):
    P = _pipeline()
    L, B = 93, 12
    plan = P.plan_transfers(L, B, chunks)
    held = {}
    ti = 0
    for idx, (rank, first, last) in enumerate(chunks):
        h = held.setdefault(rank, {"blocks": set(), "emb": idx == 0})
        if idx > 0 and chunks[idx - 1][0] != rank:
            t = plan[ti]
            ti += 1
            assert (t.src_rank, t.dst_rank, t.layer) == (chunks[idx - 1][0], rank, first)
            assert not (set(t.blocks) & h["blocks"]), "a cached block was sent again"
            h["blocks"] |= set(t.blocks)
            h["emb"] = h["emb"] or t.embedding
            # the open partial sum is sent exactly when `first` is inside a block
            assert (t.partial is not None) == ((first - 1) % B != 0)
        # every source layer `first` reads (Eq. 10) is now on this rank
        for e in O.value_list(first, B, L):
            if e[0] == "embed":
                assert h["emb"]
            elif e[0] == "block":
                assert e[1] in h["blocks"]
        h["blocks"] |= set(range(1, P.completed_blocks(last, B, L) + 1))
    assert ti == len(plan)


def test_plan_sizes_k3():
    P = _pipeline()
    plan = P.plan_transfers(93, 12, CONTIGUOUS)
    assert len(plan) == 1
    t = plan[0]
    # layer 48 is the last of block 4: blocks 1-3 complete, partial = layers 37..47
    assert t.embedding and t.blocks == [1, 2, 3] and t.partial == (37, 47) and t.rows() == 5
    assert P.full_attnres_rows(93, CONTIGUOUS) == 48      # h_0 + 47 layer outputs
    inter = P.plan_transfers(93, 12, INTERLEAVED)
    # rank 0's second chunk (layers 46..) already holds block 1; receives 2, 3 and the partial
    assert inter[1].dst_rank == 0 and not inter[1].embedding and inter[1].blocks == [2, 3]
    assert inter[1].partial == (37, 45)
    # rank 1's second chunk (71..) holds blocks 1..3 from before: receives 4, 5 only
    assert inter[2].blocks == [4, 5] and inter[2].partial == (61, 70)
    total = sum(t.rows() for t in inter)
    assert total < P.full_attnres_rows(93, INTERLEAVED)


def _run_chunk(first, last, L, B, h0, blocks, part, W, fn):
    """Layers first..last (and the final aggregation when last == L) from the
    state this rank holds: exact fp64, partial sums added in layer order."""
    for layer in range(first, last + 1):
        n = (layer - 1) // B + 1
        srcs = [h0] + [blocks[k] for k in range(1, n)] + ([part] if part is not None else [])
        assert len(srcs) == O.num_sources(layer, B, L)
        r, _ = O.depth_attention(np.stack(srcs), W[layer - 1])
        v = fn(layer, r)
        part = v if part is None else part + v
        if layer % B == 0 or layer == L:
            blocks[n] = part
            part = None
    final = None
    if last == L:
        N = O.num_blocks(L, B)
        final, _ = O.depth_attention(np.stack([h0] + [blocks[k] for k in range(1, N + 1)]), W[L])
    return part, final


def _stack_inputs(L, T, d, seed=3):
    rng = np.random.default_rng(seed)
    h0 = rng.standard_normal((T, d))
    W = rng.standard_normal((L + 1, d)) / np.sqrt(d)
    G = rng.standard_normal((L, d))
    Sc = rng.uniform(0.05, 0.2, size=(L, d))
    return h0, W, lambda l, x: O.synthetic_layer(x, G[l - 1], Sc[l - 1])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, chunks, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    P = _pipeline()
    L, B, T, d = 93, 12, 3, 16
    h0_full, W, fn = _stack_inputs(L, T, d)
    plan = P.plan_transfers(L, B, chunks)
    h0 = h0_full if rank == chunks[0][0] else None
    blocks, part, sent_rows = {}, None, 0
    ti = 0
    result = None
    for idx, (r, first, last) in enumerate(chunks):
        if idx > 0 and chunks[idx - 1][0] != r:
            t = plan[ti]
            ti += 1
            bufs = ([("h0", None)] if t.embedding else []) + [("b", k) for k in t.blocks] + \
                   ([("p", None)] if t.partial else [])
            for kind, k in bufs:
                if rank == t.src_rank:
                    x = h0 if kind == "h0" else (blocks[k] if kind == "b" else part)
                    dist.send(torch.from_numpy(np.ascontiguousarray(x)), dst=t.dst_rank)
                    sent_rows += 1
                elif rank == t.dst_rank:
                    buf = torch.empty((T, d), dtype=torch.float64)
                    dist.recv(buf, src=t.src_rank)
                    x = buf.numpy()
                    if kind == "h0":
                        h0 = x
                    elif kind == "b":
                        blocks[k] = x
                    else:
                        part = x
            if rank == t.src_rank:
                part = None          # the open partial sum moved on with the chunk
        if r == rank:
            part, final = _run_chunk(first, last, L, B, h0, blocks, part, W, fn)
            if final is not None:
                result = final
    if result is not None:
        queue.put((rank, result, sent_rows))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("chunks", [CONTIGUOUS, INTERLEAVED])
def test_two_rank_pipeline_reproduces_the_oracle(chunks):
    queue = mp.get_context("spawn").SimpleQueue()
    mp.spawn(_worker, args=(2, _free_port(), chunks, queue), nprocs=2, join=True)
    rank, final, _ = queue.get()
    assert rank == chunks[-1][0]
    h0, W, fn = _stack_inputs(93, 3, 16)
    ref = O.block_stack_forward(h0, W, fn, 93, 12)
    assert np.array_equal(final, ref.r[-1])
