"""GPU parity of the Block AttnRes stack backward (StackBackward: block-wise
recompute + attnres_aggregate_backward with accumulation) against the fp64
oracle's reverse sweep over the value lists, through the C ABI.

fp32 storage throughout, so the only differences are fp32 rounding: every
entry of dh0 and dW is compared to the oracle relative to its row's scale
(max |ref| over that token of dh0, that layer of dW).  Bound: the gradients
are sums over at most L+1 layer backwards, each a handful of fp32 dot
products of length d (relative error ~ sqrt(d) * 2^-24 ~ 5e-6 at d = 7168)
and a sum over T tokens for dW; errors of independent sign compound as the
square root of the depth (sqrt(94) ~ 10): 1e-4 of the row scale covers it
with margin, and a wrong source, range or sign moves entries by O(1) of it.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def A():
    import depth_wise_attention_block_gb300 as A
    return A


def _check_rows(got, ref, name):
    got = got.double().cpu().numpy()
    scale = np.abs(ref).max(axis=1, keepdims=True) + 1e-30
    err = (np.abs(got - ref) / scale).max()
    assert err <= TOL, f"{name}: worst error {err:.3g} of the row scale"
    return err


def _run(A, L, B, T, d, seed, dtype=torch.float32):
    from depth_wise_attention_block_gb300.stack import StackBackward, StackForward
    stk = W.stack(T=T, d=d, num_layers=L, block_size=B, seed=seed, device="cuda", dtype=dtype)
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    dr = torch.randn((T, d), generator=g, device="cuda").to(dtype)
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, L, B, keep_weights=False)
    fwd.run()
    bwd = StackBackward(fwd)
    dh0, dW = bwd.run(dr)
    torch.cuda.synchronize()
    return stk, dr, dh0, dW, bwd


@pytest.mark.parametrize("L,B,T,d", [
    (7, 3, 33, 3584),     # ring kernels (one vector per thread), three blocks, the last incomplete
    (14, 4, 17, 1000),    # 250 vectors per row: ragged last warp
    (5, 1, 9, 256),       # block size 1: Full AttnRes
    (6, 12, 5, 7168),     # one block: every layer reads [h0, partial]; fp32 rows of d = 7168 (plain loads)
    (1, 12, 4, 64),       # one layer: the final aggregation reads [h0, v1]
    (8, 4, 6, 128),       # two whole blocks, the last layer ends the second
])
def test_stack_backward_matches_the_oracle(A, L, B, T, d):
    stk, dr, dh0, dW, _ = _run(A, L, B, T, d, seed=50 + L + B)
    to = lambda t: t.double().cpu().numpy()
    rdh0, rdW = O.block_stack_backward(to(stk.h0), to(stk.W), to(stk.G), to(stk.Sc), L, B, to(dr))
    e1 = _check_rows(dh0, rdh0, "dh0")
    e2 = _check_rows(dW, rdW, "dW")
    print(f"L={L} B={B} T={T} d={d}: dh0 {e1:.3g}, dW {e2:.3g} of the row scale")


def test_stack_backward_k3_layout_93_layers(A):
    L, B, T, d = 93, 12, 8, 3584
    stk, dr, dh0, dW, _ = _run(A, L, B, T, d, seed=91)
    to = lambda t: t.double().cpu().numpy()
    rdh0, rdW = O.block_stack_backward(to(stk.h0), to(stk.W), to(stk.G), to(stk.Sc), L, B, to(dr))
    e1 = _check_rows(dh0, rdh0, "dh0")
    e2 = _check_rows(dW, rdW, "dW")
    print(f"K3 93 layers: dh0 {e1:.3g}, dW {e2:.3g} of the row scale")


def test_stack_backward_graph_replay_equals_eager(A):
    L, B, T, d = 9, 4, 16, 3584
    stk, dr, dh0, dW, bwd = _run(A, L, B, T, d, seed=7)
    e_dh0, e_dW = dh0.clone(), dW.clone()
    bwd.capture(dr)
    bwd.run()
    torch.cuda.synchronize()
    assert torch.equal(bwd.dh0, e_dh0) and torch.equal(bwd.dW, e_dW)


def test_stack_backward_bf16_tracks_fp32(A):
    # bf16 storage keeps gradients in bf16 too (one dtype per call): not
    # held to the fp32 bound, but it must follow the fp32 gradients closely
    L, B, T, d = 20, 12, 16, 7168
    _, _, dh0_32, dW_32, _ = _run(A, L, B, T, d, seed=13)
    _, _, dh0_16, dW_16, _ = _run(A, L, B, T, d, seed=13, dtype=torch.bfloat16)
    rel = lambda a, b: ((a.float() - b.float()).norm() / b.float().norm()).item()
    assert torch.isfinite(dW_16).all() and torch.isfinite(dh0_16.float()).all()
    assert rel(dW_16, dW_32) < 5e-2 and rel(dh0_16, dh0_32) < 5e-2, (rel(dW_16, dW_32), rel(dh0_16, dh0_32))
