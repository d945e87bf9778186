"""Pipeline-parallel transfer plan for Block AttnRes state.

Under pipeline parallelism a layer's depth sources may have been produced on
earlier stages.  Kimi K3 chaptered tutorial, ch. 4.2 (Full AttnRes costs
cross-stage traffic of all layer outputs) and ch. 4.6 (Block AttnRes uses
cache-based pipeline communication that sends only newly produced blocks):
a stage starting at layer l needs the embedding h_0, every block sum
completed before l, and the current block's partial sum if l is not the
first layer of its block.  A receiver keeps (caches) what it was sent, so
with interleaved (virtual) stages a rank that runs several layer chunks is
only sent the blocks completed since its previous chunk.

plan_transfers is host logic: it says which [T, d] buffers cross which
boundary.  transfer_buffers names those buffers in a stage's AttnResState
(the same positions on the sending and the receiving side), and hand_off
moves them between two stages held by one process on one GPU, one device
copy per buffer, then resumes the receiver.  Between GPUs the transport is
the caller's (NCCL send / recv of the same buffers, in the same order).
"""
from __future__ import annotations

from dataclasses import dataclass, field


def _num_blocks(L: int, B: int) -> int:
    return -(-L // B)


def completed_blocks(folded: int, B: int, L: int) -> int:
    """Blocks whose sums are complete once layer outputs v_1..v_folded exist."""
    if folded <= 0:
        return 0
    n = (folded - 1) // B + 1
    return n if (folded % B == 0 or folded == L) else n - 1


def partial_range(folded: int, B: int, L: int) -> tuple[int, int] | None:
    """Layers summed in the open partial sum after v_1..v_folded, or None."""
    if folded <= 0:
        return None
    n = (folded - 1) // B + 1
    if folded % B == 0 or folded == L:
        return None
    return ((n - 1) * B + 1, folded)


@dataclass
class Transfer:
    """What crosses one stage boundary (into the chunk starting at `layer`)."""
    src_rank: int
    dst_rank: int
    layer: int                               # first layer the receiver runs
    embedding: bool                          # h_0 (sent once per receiver)
    blocks: list[int] = field(default_factory=list)   # block sums b_k sent
    partial: tuple[int, int] | None = None             # open partial sum (layers first..last)

    def rows(self) -> int:
        """[T, d] buffers sent."""
        return int(self.embedding) + len(self.blocks) + (1 if self.partial else 0)


def plan_transfers(num_layers: int, block_size: int, chunks: list[tuple[int, int, int]]) -> list[Transfer]:
    """Transfers for a forward over layer chunks run in order.

    chunks: (rank, first_layer, last_layer) in execution order, covering
    1..num_layers contiguously (the final output aggregation runs on the
    rank of the last chunk).  Every rank caches what it was sent or
    produced; a boundary sends the receiver only the block sums it lacks,
    plus the open partial sum when the chunk starts inside a block.
    """
    L, B = num_layers, block_size
    expect = 1
    for _, f, l in chunks:
        if f != expect or l < f:
            raise ValueError("chunks must cover 1..L contiguously in order")
        expect = l + 1
    if expect != L + 1:
        raise ValueError("chunks must end at layer L")
    held: dict[int, set] = {}      # rank -> block indices it holds
    has_embedding: dict[int, bool] = {}
    out: list[Transfer] = []
    prev_rank = None
    for idx, (rank, first, last) in enumerate(chunks):
        held.setdefault(rank, set())
        if idx == 0:
            has_embedding[rank] = True          # the first stage computes h_0
        elif prev_rank != rank:
            need = set(range(1, completed_blocks(first - 1, B, L) + 1))
            t = Transfer(prev_rank, rank, first, embedding=not has_embedding.get(rank, False),
                         blocks=sorted(need - held[rank]), partial=partial_range(first - 1, B, L))
            out.append(t)
            held[rank] |= need
            has_embedding[rank] = True
        # blocks completed inside this chunk are now held by `rank`
        held[rank] |= set(range(1, completed_blocks(last, B, L) + 1))
        prev_rank = rank
    return out


def full_attnres_rows(num_layers: int, chunks: list[tuple[int, int, int]]) -> int:
    """Rows Full AttnRes would send across the same boundaries without
    caching: every earlier layer output plus the embedding."""
    rows = 0
    prev = None
    for idx, (rank, first, _) in enumerate(chunks):
        if idx > 0 and rank != prev:
            rows += first  # h_0 and v_1 .. v_{first-1}
        prev = rank
    return rows


def transfer_buffers(t: Transfer, state) -> list:
    """The buffers of a stage's AttnResState that transfer `t` moves, in
    order: h_0 (if sent), the block sums b_k of t.blocks, the open partial
    sum (if sent).  The sender reads them after its last layer (its chunk
    ends by folding that layer's output), the receiver writes them into its
    own state at the same positions."""
    out = [state.h0] if t.embedding else []
    out += [state.block_reps[k - 1] for k in t.blocks]
    if t.partial is not None:
        out.append(state.partial)
    return out


def hand_off(t: Transfer, src_state, dst_state, stream=None) -> int:
    """Move transfer `t` from one stage's state to another's when both live
    in this process on one GPU: one device-to-device copy per buffer (on
    `stream`, default the current one), then the receiver resumes at layer
    t.layer - 1.  Returns the bytes copied."""
    import torch
    src, dst = transfer_buffers(t, src_state), transfer_buffers(t, dst_state)
    ctx = torch.cuda.stream(stream) if stream is not None else None
    if ctx is not None:
        ctx.__enter__()
    try:
        for a, b in zip(src, dst):
            b.copy_(a, non_blocking=True)
    finally:
        if ctx is not None:
            ctx.__exit__(None, None, None)
    dst_state.resume(t.layer - 1)
    return sum(a.numel() * a.element_size() for a in src)
