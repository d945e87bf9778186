"""Pipeline-parallel hand-off through the library, on one GPU.

A 93-layer stack is split into layer chunks run by two "ranks" (two stack
states with their own buffers; Kimi K3 chaptered tutorial, ch. 4.6:
cache-based pipeline communication sends a later stage only the blocks
completed since it last received, plus the open partial sum).  At every
boundary exactly the buffers pipeline.plan_transfers names are copied from
the sender's state into the receiver's (one device copy per buffer), the
receiver resumes its state at the boundary (attnres_state_resume) and runs
on.  The result must equal the uninterrupted single-state run bit for bit,
and, with fp32 storage, the fp64 oracle at the fp32 bars.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests.parity import A_ATOL, R_F32_RTOL, to64

pytestmark = pytest.mark.gpu

CONTIGUOUS = [(0, 1, 47), (1, 48, 93)]                       # boundary inside block 4
INTERLEAVED = [(0, 1, 20), (1, 21, 45), (0, 46, 70), (1, 71, 93)]
BLOCK_ALIGNED = [(0, 1, 36), (1, 37, 60), (0, 61, 93)]       # boundaries at block ends: no partial sum sent


@pytest.fixture(scope="module")
def A():
    import depth_wise_attention_block_gb300 as A
    return A


def _pipelined(stk, chunks):
    from depth_wise_attention_block_gb300 import pipeline as P
    from depth_wise_attention_block_gb300.stack import StackForward
    L, B = stk.num_layers, stk.block_size
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ranks = {}
    for rank in sorted({c[0] for c in chunks}):
        # only the first stage is given the embedding; the others get an
        # empty buffer that the hand-off fills
        h0 = stk.h0 if rank == chunks[0][0] else torch.full_like(stk.h0, float("nan"))
        ranks[rank] = StackForward(h0, stk.W, stk.G, stk.Sc, L, B, dev_err=err)
        for b in ranks[rank].state.block_reps + [ranks[rank].state.partial]:
            b.fill_(float("nan"))       # nothing a stage did not compute or receive is readable
    plan = iter(P.plan_transfers(L, B, chunks))
    sent = 0
    weights = {}
    for idx, (rank, first, last) in enumerate(chunks):
        if idx > 0 and chunks[idx - 1][0] != rank:
            t = next(plan)
            sent += P.hand_off(t, ranks[t.src_rank].state, ranks[t.dst_rank].state)
        f = ranks[rank]
        f.run_chunk(first, last)
        for l in range(first, last + 2 if last == L else last + 1):
            weights[l] = f.weights[l - 1].clone()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return ranks[chunks[-1][0]].r.clone(), weights, sent


def _whole(stk):
    from depth_wise_attention_block_gb300.stack import StackForward
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, stk.num_layers, stk.block_size)
    fwd.run()
    torch.cuda.synchronize()
    return fwd


@pytest.mark.parametrize("chunks", [CONTIGUOUS, INTERLEAVED, BLOCK_ALIGNED], ids=["contiguous", "interleaved",
                                                                                 "block_aligned"])
@pytest.mark.parametrize("dtype,d", [(torch.float32, 3584), (torch.bfloat16, 7168)])
def test_pipelined_stack_equals_the_whole_stack(A, chunks, dtype, d):
    from depth_wise_attention_block_gb300 import pipeline as P
    stk = W.stack(T=16, d=d, num_layers=93, block_size=12, seed=57, device="cuda", dtype=dtype)
    r, weights, sent = _pipelined(stk, chunks)
    ref = _whole(stk)
    assert torch.equal(r, ref.r)
    for l, a in weights.items():
        assert torch.equal(a, ref.weights[l - 1]), f"layer {l}"
    row = 16 * d * stk.h0.element_size()
    assert sent == row * sum(t.rows() for t in P.plan_transfers(93, 12, chunks))
    if dtype == torch.float32:
        # against the fp64 oracle (fp32 storage rounding) at the fp32 bars
        G, Sc = to64(stk.G), to64(stk.Sc)
        tr = O.block_stack_forward(to64(stk.h0), to64(stk.W), lambda l, x: O.synthetic_layer(x, G[l - 1], Sc[l - 1]),
                                   93, 12, store=O.round_fp32)
        for l, a in weights.items():
            assert np.abs(to64(a) - tr.a[l - 1]).max() <= A_ATOL, f"layer {l}"
        M = np.abs(np.stack(tr.final_sources)).max(axis=(0, 2))[:, None]
        assert (np.abs(to64(r) - tr.r[-1]) <= R_F32_RTOL * (np.abs(tr.r[-1]) + M)).all()
