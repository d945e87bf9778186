"""Per-layer parity of the bf16 stacks at the single-layer bars (teacher forcing).

A free-running bf16 stack drifts from the oracle by one-ulp storage flips
that compound over 93 layers, so its whole-stack check needs a looser weight
bar.  Here every layer of the GPU stack is checked on its own instead: the
oracle is given the bytes the GPU's stack state held for that layer (h_0,
the stored block sums b_k, the stored partial sum) and must agree with the
layer's weights within 1e-5 and with its stored r within the bf16 bar
(one ulp + 1e-3 of the token's largest source value).  The oracle stays a
pure fp64 function of its arguments; only its inputs come from the run.

Also per layer: every partial sum or block sum the step wrote equals
round_bf16(stored partial + stored F) bit for bit (the bookkeeping of Kimi
K3 chaptered tutorial, ch. 4.3, Eq. 10, with one rounding at the store), and
the stand-in body's output is within one ulp of the exact body on the
stored r.

The same for the stack backward: each layer's attnres_aggregate_backward
call is checked against the oracle's backward on the bytes that call read
(its sources, its incoming gradient) and on the gradient buffers as they
were before it (the call accumulates into them).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests.parity import A_ATOL, R_BF16_MABS, to64, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import depth_wise_attention_block_gb300 as A
    return A


def _sources_of(l, L, B, h0, blocks, partial_at):
    """Eq. 10's sources of layer l from the stored rows: h_0, b_1..b_{n-1},
    and the partial sum the step of layer l left (i >= 2); the final
    aggregation (l = L+1) reads h_0 and every block sum."""
    if l == L + 1:
        return [h0] + blocks
    n, i = O.block_index(l, B), O.position_in_block(l, B)
    return [h0] + blocks[: n - 1] + ([partial_at[l]] if i >= 2 else [])


def _teacher_forced_forward(A, stk, tokens, schedule="single"):
    from depth_wise_attention_block_gb300.stack import StackForward
    L, B = stk.num_layers, stk.block_size
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, L, B, dev_err=err, schedule=schedule, two_phase_from=5)
    r_at, F_at, partial_at = {}, {}, {}

    def hook(l, f):
        r_at[l] = to64(f.r[tokens])
        if l <= L:
            F_at[l] = to64(f.F[tokens])
            partial_at[l] = to64(f.state.partial[tokens])

    fwd.run(on_layer=hook)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    h0 = to64(stk.h0[tokens])
    blocks = [to64(b[tokens]) for b in fwd.state.block_reps]
    Wq, G, Sc = to64(stk.W), to64(stk.G), to64(stk.Sc)
    worst_a, worst_r = 0.0, 0.0
    for l in range(1, L + 2):
        srcs = _sources_of(l, L, B, h0, blocks, partial_at)
        r_ref, a_ref = O.depth_attention(np.stack(srcs), Wq[l - 1])
        a = to64(fwd.weights[l - 1][tokens])
        ea = float(np.abs(a - a_ref).max())
        assert ea <= A_ATOL, f"layer {l}: weights off by {ea:.3g}"
        M = np.abs(np.stack(srcs)).max(axis=(0, 2))[:, None]
        bound = ulp_bf16(r_ref) + R_BF16_MABS * M
        er = np.abs(r_at[l] - r_ref) / bound
        assert er.max() <= 1.0, f"layer {l}: r off by {er.max():.3g} x the bf16 bar"
        worst_a, worst_r = max(worst_a, ea), max(worst_r, float(er.max()))
        if l >= 2:
            # the row the step of layer l wrote: partial + F_{l-1} (or F_{l-1}
            # alone at a block's second layer), rounded once
            p = l - 1
            first = (O.block_index(p, B) - 1) * B + 1
            prev = partial_at[p] if p > first else 0.0
            formed = O.round_bf16(prev + F_at[p])
            ends = p % B == 0 or p == L
            stored = blocks[O.block_index(p, B) - 1] if ends else partial_at[l]
            assert np.array_equal(stored, formed), f"layer {l}: the folded row is not round(partial + F)"
        if l <= L:
            F_ref = O.synthetic_layer(r_at[l], G[l - 1], Sc[l - 1])
            assert (np.abs(F_at[l] - F_ref) <= ulp_bf16(F_ref)).all(), f"layer {l}: stand-in body"
    return worst_a, worst_r


def test_decode_stack_T64_every_layer_every_token(A):
    # 93-layer bf16 stack, T = 64 (one decode step for 64 sequences), seed 3
    stk = W.stack_T64(device="cuda")
    wa, wr = _teacher_forced_forward(A, stk, torch.arange(64, device="cuda"))
    print(f"decode T=64 per layer: worst weight error {wa:.3g}, worst r {wr:.3g} x bar")


@pytest.mark.parametrize("schedule", ["two_phase", "hybrid"])
def test_decode_stack_T64_two_phase_every_layer(A, schedule):
    stk = W.stack_T64(device="cuda")
    wa, wr = _teacher_forced_forward(A, stk, torch.arange(64, device="cuda"), schedule=schedule)
    print(f"decode T=64 {schedule} per layer: worst weight error {wa:.3g}, worst r {wr:.3g} x bar")


def test_full_attnres_bf16_stack_every_layer(A):
    # block size 1 (Full AttnRes): layer l aggregates all l earlier outputs,
    # up to 94 sources at the final aggregation -- the multi-group kernel
    # fused into the stack steps, every layer at the single-layer bars
    stk = W.stack(T=32, num_layers=93, block_size=1, seed=7, device="cuda")
    wa, wr = _teacher_forced_forward(A, stk, torch.arange(32, device="cuda"))
    print(f"Full AttnRes bf16 T=32 per layer: worst weight error {wa:.3g}, worst r {wr:.3g} x bar")


@pytest.mark.parametrize("schedule", ["single", "hybrid"])
def test_prefill_stack_T2048_every_layer_sampled_tokens(A, schedule):
    # 93-layer bf16 stack, T = 2048, seed 2; tokens at the persistent CTAs'
    # boundaries (token t goes to CTA t mod 152: CTAs 0..71 take 14 tokens,
    # 72..151 take 13; in the inter-block pass tokens 1976..2047 are split in
    # two query halves) plus a seeded random sample, 64 in all.  Hybrid: the
    # blocks from the fifth on run two-phase.
    stk = W.stack_T2048(device="cuda")
    edge = [0, 1, 71, 72, 151, 152, 1975, 1976, 2046, 2047]
    g = torch.Generator().manual_seed(2048)
    rest = [t for t in torch.randperm(2048, generator=g).tolist() if t not in edge][: 64 - len(edge)]
    tokens = torch.tensor(sorted(edge + rest), device="cuda")
    wa, wr = _teacher_forced_forward(A, stk, tokens, schedule=schedule)
    print(f"prefill T=2048 {schedule} per layer ({tokens.numel()} tokens): worst weight error {wa:.3g}, "
          f"worst r {wr:.3g} x bar")


@pytest.mark.parametrize("schedule", ["single", "hybrid"])
def test_stack_backward_bf16_every_layer_call(A, schedule):
    # 93-layer bf16 stack backward (block-wise recompute), T = 32, d = 7168:
    # each attnres_aggregate_backward call against the oracle's backward on
    # the bytes it read; source gradients within one bf16 ulp + 1e-3 of the
    # token's largest condition scale (the bar of the single-layer backward
    # tests), grad_w within 1e-5 of its condition scale.  The forward's
    # block sums (all the backward keeps) come from either schedule.
    from depth_wise_attention_block_gb300.stack import StackBackward, StackForward
    L, B, T, d = 93, 12, 32, 7168
    stk = W.stack(T=T, d=d, num_layers=L, block_size=B, seed=17, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(18)
    dr_out = torch.randn((T, d), generator=g, device="cuda").to(torch.bfloat16)
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, L, B, keep_weights=False, schedule=schedule,
                       two_phase_from=5)
    fwd.run()
    bwd = StackBackward(fwd)
    Wq = to64(stk.W)
    seen = {"calls": 0, "worst_h": 0.0, "worst_w": 0.0}
    before = {}

    def hook(layer, srcs, grad_r, grads, grad_w, accumulate, phase):
        if phase == "before":
            before["srcs"] = np.stack([to64(s) for s in srcs])
            before["dr"] = to64(grad_r)
            before["g"] = [to64(x) for x in grads] if accumulate else [0.0] * len(grads)
            return
        dH, dw = O.depth_attention_backward(before["srcs"], Wq[layer - 1], before["dr"])
        dHs, dws = O.depth_attention_backward_scales(before["srcs"], Wq[layer - 1], before["dr"])
        ew = np.abs(to64(grad_w) - dw) / (1e-5 * dws + 1e-30)
        assert ew.max() <= 1.0, f"layer {layer}: grad_w off by {ew.max():.3g} x its bar"
        for s, x in enumerate(grads):
            want = before["g"][s] + dH[s]
            bound = ulp_bf16(want) + 1e-3 * dHs[s].max(axis=1, keepdims=True)
            eh = np.abs(to64(x) - want) / bound
            assert eh.max() <= 1.0, f"layer {layer}, source {s}: gradient off by {eh.max():.3g} x its bar"
            seen["worst_h"] = max(seen["worst_h"], float(eh.max()))
        seen["worst_w"] = max(seen["worst_w"], float(ew.max()))
        seen["calls"] += 1

    bwd.run(dr_out, on_call=hook)
    torch.cuda.synchronize()
    assert seen["calls"] == L + 1
    print(f"bf16 stack backward, {seen['calls']} calls: worst source gradient {seen['worst_h']:.3g} x bar, "
          f"grad_w {seen['worst_w']:.3g} x bar")
