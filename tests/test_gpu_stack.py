"""GPU parity of the fused stack path (attnres_layer_step + the block
bookkeeping) against the fp64 oracle run with the same storage rounding.

The oracle runs the whole stack on its own (free-running): it never sees a
GPU result.  Per token the stack is independent of every other token, so at
full size the oracle runs on sampled tokens only.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests.parity import A_ATOL, R_BF16_MABS, R_F32_RTOL, STACK_BF16_A_ATOL, to64, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    import depth_wise_attention_block_gb300 as A
    return A


def _oracle_stack(stk: W.Stack, tokens=None, store=O.round_bf16):
    h0 = to64(stk.h0 if tokens is None else stk.h0[tokens])
    G, Sc, Wq = to64(stk.G), to64(stk.Sc), to64(stk.W)
    fn = lambda l, x: O.synthetic_layer(x, G[l - 1], Sc[l - 1])
    return O.block_stack_forward(h0, Wq, fn, stk.num_layers, stk.block_size, store=store)


def _gpu_stack(A, stk: W.Stack, graph=False, schedule="single", two_phase_from=5):
    from depth_wise_attention_block_gb300.stack import StackForward
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, stk.num_layers, stk.block_size, dev_err=err,
                       schedule=schedule, two_phase_from=two_phase_from)
    if graph:
        fwd.capture()
    fwd.run()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return fwd


def _layer_bar(ref_sources, r_ref, dtype):
    """Per-element bound of a stack output, at the scale M_t = max_{s,c}
    |h_s[t, c]| of the token's sources (errors of a stack are absolute at
    that scale: they flow in from earlier layers' outputs):
    fp32 storage: 1e-5 (|ref| + M_t); bf16 storage: ulp_bf16(ref) + 1e-3 M_t."""
    M = np.abs(np.stack(ref_sources)).max(axis=(0, 2))[:, None]
    if dtype == torch.float32:
        return R_F32_RTOL * (np.abs(r_ref) + M)
    return ulp_bf16(r_ref) + R_BF16_MABS * M


def _check_stack(fwd, tr, tokens, dtype, weight_tol, check_blocks=True):
    """Every layer's weights, the final output and (optionally) the resident
    block representations against the oracle trace.  Block sums of a long
    free-running bf16 stack add up a dozen layer outputs that each carry
    their own rounding flips, so the per-element bar is only applied to them
    in fp32 storage and in short bf16 stacks."""
    worst_a, worst_r = 0.0, 0.0
    L = fwd.L
    for l in range(1, L + 2):
        a = to64(fwd.weights[l - 1][tokens])
        worst_a = max(worst_a, float(np.abs(a - tr.a[l - 1]).max()))
    assert worst_a <= weight_tol, f"weights off by {worst_a:.3g}"
    r = to64(fwd.r[tokens])
    bound = _layer_bar(tr.final_sources, tr.r[-1], dtype)
    err = np.abs(r - tr.r[-1])
    worst_r = float((err / bound).max())
    assert worst_r <= 1.0, f"final output off by {worst_r:.3g} x the bound"
    # the resident block representations after the forward
    for k, b in enumerate(fwd.state.block_reps if check_blocks else []):
        ref = tr.final_sources[k + 1]
        bb = _layer_bar(tr.final_sources, ref, dtype)
        assert (np.abs(to64(b[tokens]) - ref) <= bb).all(), f"block rep {k + 1}"
    return worst_a, worst_r


@pytest.mark.parametrize("L,B,T,d,dtype", [
    (7, 3, 6, 64, torch.bfloat16),      # ring kernel, 3 blocks, the last incomplete
    (12, 1, 5, 40, torch.float32),      # block size 1 = Full AttnRes; S reaches 13 (generic kernel)
    (9, 4, 7, 7168, torch.bfloat16),    # K3 width, ring, 2 vectors per thread
    (5, 9, 3, 24, torch.float32),       # one block holds every layer
    (1, 12, 4, 64, torch.float32),      # one layer: the final aggregation reads [h0, v1]
    (12, 12, 5, 256, torch.bfloat16),   # the block ends exactly at the last layer
    (2, 1, 3, 16, torch.bfloat16),      # block size 1, two layers
])
def test_tiny_stacks_every_layer(A, L, B, T, d, dtype):
    stk = W.stack(T=T, d=d, num_layers=L, block_size=B, seed=31 + L + B, device="cuda", dtype=dtype)
    fwd = _gpu_stack(A, stk)
    store = O.round_bf16 if dtype == torch.bfloat16 else O.round_fp32
    tr = _oracle_stack(stk, store=store)
    tol = A_ATOL if dtype == torch.float32 else STACK_BF16_A_ATOL
    _check_stack(fwd, tr, slice(None), dtype, tol)


@pytest.mark.parametrize("d", [3584, 7168])
def test_k3_layout_fp32_storage_93_layers(A, d):
    # the full 93-layer / 12-layer-block bookkeeping at the fp32 bars (no bf16
    # rounding flips to compound); d=3584 fp32 runs the bulk-copy ring kernel
    # (896 vectors per row), d=7168 fp32 the generic kernel
    stk = W.stack(T=64, d=d, seed=41, device="cuda", dtype=torch.float32)
    fwd = _gpu_stack(A, stk)
    tr = _oracle_stack(stk, store=O.round_fp32)
    wa, wr = _check_stack(fwd, tr, slice(None), torch.float32, A_ATOL)
    print(f"fp32 93-layer stack d={d}: worst weight error {wa:.3g}, worst output error {wr:.3g} x bound")


@pytest.mark.parametrize("d", [3584, 7168])
def test_full_attnres_fp32_storage_93_layers(A, d):
    # block size 1 = Full AttnRes: layer l aggregates all l earlier outputs
    # (up to 94 sources: the multi-group ring kernel at d=3584, the generic
    # kernel at d=7168 fp32), at the fp32 bars over all 93 layers
    stk = W.stack(T=16, d=d, num_layers=93, block_size=1, seed=43, device="cuda", dtype=torch.float32)
    fwd = _gpu_stack(A, stk)
    assert fwd.S[-1] == 94
    tr = _oracle_stack(stk, store=O.round_fp32)
    wa, wr = _check_stack(fwd, tr, slice(None), torch.float32, A_ATOL)
    print(f"Full AttnRes fp32 93 layers d={d}: worst weight error {wa:.3g}, worst output error {wr:.3g} x bound")


def test_full_attnres_bf16_93_layers(A):
    stk = W.stack(T=16, d=7168, num_layers=93, block_size=1, seed=44, device="cuda")
    fwd = _gpu_stack(A, stk, graph=True)
    tr = _oracle_stack(stk)
    wa, wr = _check_stack(fwd, tr, slice(None), torch.bfloat16, STACK_BF16_A_ATOL, check_blocks=False)
    print(f"Full AttnRes bf16 93 layers: worst weight error {wa:.3g}, worst output error {wr:.3g} x bound")


@pytest.mark.parametrize("schedule,T,dtype", [("two_phase", 64, torch.bfloat16), ("hybrid", 300, torch.bfloat16),
                                              ("two_phase", 33, torch.float32)])
def test_first_layer_from_the_pass_changes_no_bit(A, schedule, T, dtype):
    """A two-phase block's first layer written by the inter-block pass
    (out_r0, out_weights0) gives the bits of its merge step."""
    from depth_wise_attention_block_gb300.stack import StackForward
    d = 7168 if dtype == torch.bfloat16 else 1024
    stk = W.stack(T=T, d=d, num_layers=30, block_size=6, seed=11 + T, device="cuda", dtype=dtype)
    outs = []
    for own in (True, False):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, 30, 6, dev_err=err, schedule=schedule, two_phase_from=2,
                           first_layer_from_pass=own)
        fwd.run()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((fwd.r.clone(), torch.cat(fwd.weights, dim=1).clone(),
                     [b.clone() for b in fwd.state.block_reps]))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert all(torch.equal(x, y) for x, y in zip(outs[0][2], outs[1][2]))


@pytest.mark.parametrize("T,L,B,dtype,graph,schedule", [
    (64, 93, 12, torch.bfloat16, True, "single"),     # the decode stack, replayed from a CUDA graph
    (64, 93, 12, torch.bfloat16, False, "single"),
    (300, 20, 4, torch.float32, True, "single"),      # two tokens per CTA on some SMs
    (5, 14, 1, torch.bfloat16, False, "single"),      # Full AttnRes layout: every step closes a block
    (64, 93, 12, torch.bfloat16, True, "hybrid"),     # the ring merges of blocks 6-8
    (300, 30, 12, torch.bfloat16, False, "two_phase"),
])
def test_early_loads_change_no_bit(A, T, L, B, dtype, graph, schedule):
    """The fused steps' and ring merges' rows that earlier kernels wrote,
    loaded before the previous kernel ends (the stack drivers' default),
    give the same bits as loads after it."""
    from depth_wise_attention_block_gb300.stack import StackForward
    stk = W.stack(T=T, d=7168 if dtype == torch.bfloat16 else 1024, num_layers=L, block_size=B, seed=90 + T + L,
                  device="cuda", dtype=dtype)
    outs = []
    for early in (True, False):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, L, B, dev_err=err, early_loads=early, schedule=schedule)
        assert bool(fwd.state.struct.flags & A.ATTNRES_STATE_EARLY_LOADS) == early
        if graph:
            fwd.capture()
        for _ in range(3):   # replays back to back: each forward's first step follows the last one's kernels
            fwd.run()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((fwd.r.clone(), torch.cat(fwd.weights, dim=1).clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("n,d,dtype,prev,in_place", [
    (3, 7168, torch.bfloat16, True, False),    # the ring kernel with the source count fixed
    (8, 7168, torch.bfloat16, False, False),   # nine sources, the partial from F alone
    (5, 7168, torch.bfloat16, True, True),     # dst is prev, updated in place
    (5, 1024, torch.float32, True, False),
    (15, 7168, torch.bfloat16, True, False),   # sixteen sources: the multi-group kernel
    (2, 1000, torch.bfloat16, True, False),    # 2000-byte rows: the plain-load kernel
    (0, 7168, torch.bfloat16, True, False),    # the partial sum is the only source
])
def test_aggregate_fold_equals_fold_then_aggregate(A, n, d, dtype, prev, in_place):
    T = 333
    g = torch.Generator(device="cuda").manual_seed(n * 7 + d)
    rows = [(torch.randn((T, d), generator=g, device="cuda") * (0.5 + k)).to(dtype) for k in range(n + 2)]
    srcs, P, F = rows[:n], rows[n], rows[n + 1]
    w = torch.randn((d,), generator=g, device="cuda") / d ** 0.5
    # reference: attnres_fold, then attnres_aggregate over [srcs, P']
    P_ref = torch.empty_like(F)
    A.attnres_fold(P if prev else None, F, P_ref)
    r_ref = torch.empty_like(F)
    a_ref = torch.empty((T, n + 1), device="cuda")
    A.attnres_aggregate(srcs + [P_ref], w, r_ref, a_ref)
    dst = P if in_place else torch.empty_like(F)
    r = torch.empty_like(F)
    a = torch.empty((T, n + 1), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # early loads are safe here: the kernels before this launch wrote all the
    # rows it reads and have completed (stream order and the signal after the wait)
    A.attnres_aggregate_fold(srcs, P if prev else None, F, dst, w, r, a, early_loads=n % 2 == 1, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(dst, P_ref) and torch.equal(r, r_ref) and torch.equal(a, a_ref)


def _random_fold_cases(n=12, seed=77):
    # seeded shapes for the fused fold: stored sources 0..127, T 1..400,
    # widths on every aggregation kernel, both dtypes, prev or not, in place
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        ns = int(rng.choice([0, 1, 2, 5, 8, 9, 12, 30, 93, 127]))
        d = int(rng.choice([8, 64, 100, 1000, 3584, 7160, 7168]))
        T = int(rng.integers(1, 401))
        dtype = [torch.bfloat16, torch.float32][int(rng.integers(2))]
        if (ns + 2) * T * d > 40_000_000:
            continue
        out.append((ns, d, T, dtype, bool(rng.integers(2)), bool(rng.integers(2))))
    return out


@pytest.mark.parametrize("n,d,T,dtype,prev,in_place", _random_fold_cases())
def test_aggregate_fold_random_shapes(A, n, d, T, dtype, prev, in_place):
    """attnres_aggregate_fold = attnres_fold + attnres_aggregate bit for bit
    on seeded shapes."""
    g = torch.Generator(device="cuda").manual_seed(n * 131 + d + T)
    rows = [(torch.randn((T, d), generator=g, device="cuda") * (0.5 + k % 5)).to(dtype) for k in range(n + 2)]
    srcs, P, F = rows[:n], rows[n], rows[n + 1]
    w = torch.randn((d,), generator=g, device="cuda") / d ** 0.5
    P_ref = torch.empty_like(F)
    A.attnres_fold(P if prev else None, F, P_ref)
    r_ref, a_ref = torch.empty_like(F), torch.empty((T, n + 1), device="cuda")
    A.attnres_aggregate(srcs + [P_ref], w, r_ref, a_ref)
    dst = P if (in_place and prev) else torch.empty_like(F)
    r, a = torch.empty_like(F), torch.empty((T, n + 1), device="cuda")
    A.attnres_aggregate_fold(srcs, P if prev else None, F, dst, w, r, a)
    torch.cuda.synchronize()
    assert torch.equal(dst, P_ref) and torch.equal(r, r_ref) and torch.equal(a, a_ref)


def test_fused_equals_unfused_bit_for_bit(A):
    L, B, T, d = 14, 4, 33, 7168
    stk = W.stack(T=T, d=d, num_layers=L, block_size=B, seed=77, device="cuda")
    fused = _gpu_stack(A, stk)
    # unfused: block_step, then aggregate over layer_sources
    st = A.AttnResState.allocate(stk.h0, L, B)
    r = torch.empty_like(stk.h0)
    F = torch.empty_like(stk.h0)
    for l in range(1, L + 2):
        if l > 1:
            A.attnres_block_step(st, F, l - 1)
        ptrs = A.attnres_layer_sources(st, l)
        bufs = {t.data_ptr(): t for t in [st.h0, st.partial] + st.block_reps}
        srcs = [bufs[p] for p in ptrs]
        a = torch.empty((T, len(srcs)), dtype=torch.float32, device="cuda")
        A.attnres_aggregate(srcs, stk.W[l - 1], r, a)
        assert torch.equal(a, fused.weights[l - 1]), f"layer {l} weights differ"
        if l <= L:
            A.attnres_synthetic_layer(r, stk.G[l - 1], stk.Sc[l - 1], F)
    torch.cuda.synchronize()
    assert torch.equal(r, fused.r)
    for b1, b2 in zip(st.block_reps, fused.state.block_reps):
        assert torch.equal(b1, b2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,d", [(300, 7168), (37, 100)])
def test_synthetic_layer_against_oracle(A, dtype, T, d):
    # The stand-in body F(x) = tanh(x g) s element by element against the
    # oracle on the same stored inputs.  fp32 storage: a few fp32 ulps of the
    # exact value.  bf16 storage (its tanh is the hardware approximation,
    # well below half a bf16 ulp): within one bf16 ulp of the exact value,
    # and nearly always its correctly rounded value.  d = 100 takes the
    # plain-load kernel, d = 7168 the vector one.
    gen = torch.Generator().manual_seed(41 + d)
    x = (torch.randn(T, d, generator=gen) * 2.0).to(dtype)
    G = torch.randn(d, generator=gen)
    Sc = 0.05 + 0.15 * torch.rand(d, generator=gen)
    out = torch.full((T, d), float("nan"), dtype=dtype, device="cuda")
    A.attnres_synthetic_layer(x.cuda(), G.cuda(), Sc.cuda(), out)
    torch.cuda.synchronize()
    ref = O.synthetic_layer(to64(x), to64(G), to64(Sc))
    got = to64(out)
    err = np.abs(got - ref)
    if dtype == torch.float32:
        assert (err <= 1e-6 * np.abs(ref) + 1e-30).all(), f"worst {float((err / np.abs(ref)).max()):.3g} relative"
    else:
        assert (err <= ulp_bf16(ref)).all(), "a bf16 output is more than one ulp from the exact value"
        off = float((got != O.round_bf16(ref)).mean())
        assert off < 0.02, f"{off:.2%} of the outputs are not the correctly rounded value"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,d,two", [(300, 7168, True), (300, 7168, False), (37, 100, True)])
def test_synthetic_layer_backward_against_oracle(A, dtype, T, d, two):
    # grad_x = (dv_a + dv_b) sech(x g)^2 g s element by element against the
    # oracle on the same stored inputs (dv_a + dv_b summed in fp32 first, as
    # the kernel does; exact for bf16 gradients).  fp32: within 1e-5 of the
    # value plus 1e-6 of the scale |dv g s| (sech^2 <= 1); bf16: within one
    # bf16 ulp of the exact value.
    gen = torch.Generator().manual_seed(43 + d)
    x = (torch.randn(T, d, generator=gen) * 2.0).to(dtype)
    G = torch.randn(d, generator=gen)
    Sc = 0.05 + 0.15 * torch.rand(d, generator=gen)
    dva = torch.randn(T, d, generator=gen).to(dtype)
    dvb = torch.randn(T, d, generator=gen).to(dtype) if two else None
    gx = torch.full((T, d), float("nan"), dtype=dtype, device="cuda")
    A.attnres_synthetic_layer_backward(x.cuda(), G.cuda(), Sc.cuda(), dva.cuda(),
                                       dvb.cuda() if two else None, gx)
    torch.cuda.synchronize()
    dv = to64(dva) + (to64(dvb) if two else 0.0)
    if dtype == torch.float32:
        dv = dv.astype(np.float32).astype(np.float64)  # the kernel's fp32 sum
    ref = O.synthetic_layer_backward(to64(x), to64(G), to64(Sc), dv)
    scale = np.abs(dv * to64(G) * to64(Sc))
    err = np.abs(to64(gx) - ref)
    if dtype == torch.float32:
        assert (err <= 1e-5 * np.abs(ref) + 1e-6 * scale).all(), f"worst {float((err / (scale + 1e-30)).max()):.3g}"
    else:
        assert (err <= ulp_bf16(ref) + 1e-6 * scale).all(), "a bf16 gradient is more than one ulp off"


def test_cuda_graph_replay_matches_eager(A):
    stk = W.stack(T=64, num_layers=20, block_size=12, seed=5, device="cuda")
    eager = _gpu_stack(A, stk)
    graphed = _gpu_stack(A, stk, graph=True)
    graphed.run()
    torch.cuda.synchronize()
    assert torch.equal(eager.r, graphed.r)
    for a1, a2 in zip(eager.weights, graphed.weights):
        assert torch.equal(a1, a2)


def test_decode_stack_T64_every_token(A):
    stk = W.stack_T64(device="cuda")
    fwd = _gpu_stack(A, stk, graph=True)
    tr = _oracle_stack(stk)
    wa, wr = _check_stack(fwd, tr, slice(None), torch.bfloat16, STACK_BF16_A_ATOL, check_blocks=False)
    print(f"decode stack T=64: worst weight error {wa:.3g}, worst output error {wr:.3g} x bound")


def test_prefill_stack_T2048_sampled_tokens(A):
    stk = W.stack_T2048(device="cuda")
    fwd = _gpu_stack(A, stk)
    tokens = torch.tensor([0, 1, 151, 152, 1000, 1023, 2046, 2047], device="cuda")
    tr = _oracle_stack(stk, tokens)
    wa, wr = _check_stack(fwd, tr, tokens, torch.bfloat16, STACK_BF16_A_ATOL, check_blocks=False)
    print(f"prefill stack T=2048: worst weight error {wa:.3g}, worst output error {wr:.3g} x bound")


def test_bytes_model_counts_k3_sources(A):
    stk = W.stack(T=8, d=64, seed=1, device="cuda")
    from depth_wise_attention_block_gb300.stack import StackForward
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, 93, 12)
    assert sum(fwd.S[:93]) == 493 and fwd.S[-1] == 9
    assert fwd.bytes_moved() > 0


# ------------------------------------------------- two-phase schedule -------

@pytest.mark.parametrize("tensor_cores", [True, False], ids=["tcgen05_logits", "cuda_cores"])
@pytest.mark.parametrize("n,Q,dtype,d", [
    (1, 12, torch.bfloat16, 7168),   # tensor cores: 128 tokens per tile, 2 tiles (the second ragged)
    (5, 3, torch.bfloat16, 7168),    # 16 tokens x 8 rows (3 zero rows), ragged last tile
    (3, 12, torch.bfloat16, 7168),   # 32 tokens x 4 rows
    (8, 12, torch.bfloat16, 7168),   # the K3 top block: 16 tokens x 8 rows
    (9, 16, torch.bfloat16, 1024),   # 8 tokens x 16 rows, 16 channel atoms, Q = 16
    (5, 12, torch.bfloat16, 1088),   # 17 channel chunks of 64: an odd count, split over CTAs
    (9, 12, torch.float32, 3584),    # fp32 sources: CUDA cores either way
    (8, 9, torch.bfloat16, 7160),    # d not a multiple of 64: CUDA cores either way
])
def test_interblock_pass_matches_the_oracle(A, n, Q, dtype, d, tensor_cores, T=150):
    from tests.parity import oracle_aggregate
    inp = W.block_bf16(T=T, d=d, seed=60 + n + Q, device="cuda", num_blocks=max(n - 2, 0), src_dtype=dtype)
    H = inp.H[:n].contiguous()
    g = torch.Generator(device="cuda").manual_seed(n)
    Wq = torch.randn((Q, d), generator=g, device="cuda") / d ** 0.5
    R = torch.empty((Q, T, d), device="cuda")
    lse = torch.empty((Q, T), device="cuda")
    Aw = torch.empty((Q, T, n), device="cuda")
    r0 = torch.empty((T, d), dtype=dtype, device="cuda")
    a0 = torch.empty((T, n), device="cuda")
    A.attnres_interblock(list(H.unbind(0)), Wq, R, lse, Aw, tensor_cores=tensor_cores, out_r0=r0, out_weights0=a0)
    torch.cuda.synchronize()
    # the first layer's outputs: query 0's row rounded (as 1 * r + 0) and its weights
    assert torch.equal(r0, (R[0] + 0.0).to(dtype)) and torch.equal(a0, Aw[0])
    uses_tc = tensor_cores and A.attnres_interblock_workspace_size(n, T, d, dtype, Q) > 0
    assert uses_tc == (tensor_cores and dtype == torch.bfloat16 and d % 64 == 0)
    for q in range(Q):
        r_ref, a_ref, l_ref = O.depth_attention_lse(to64(H), to64(Wq[q]))
        _, _, cond, M = oracle_aggregate(H, Wq[q], 1e-5)
        assert np.abs(to64(Aw[q]) - a_ref).max() <= A_ATOL
        assert (np.abs(to64(R[q]) - r_ref) <= R_F32_RTOL * (np.abs(r_ref) + cond)).all()
        assert (np.abs(to64(lse[q]) - l_ref) <= 1e-5 * (1 + np.abs(l_ref))).all()


@pytest.mark.parametrize("n", [2, 4, 6, 7, 9])
def test_interblock_every_source_count_at_k3_width(A, n):
    """The tensor-core pass at d = 7168 fixes the source count at compile
    time; the shapes above cover n = 1, 3, 5, 8, these the rest."""
    test_interblock_pass_matches_the_oracle(A, n, 12 if n % 2 else 7, torch.bfloat16, 7168, True)


def _random_interblock_cases(n_cases=12, seed=20261202):
    """Seeded shapes for the tensor-core pass: T across tile (16-128 tokens)
    and persistent-round (152) boundaries, every source count, query counts
    1..16, d any multiple of 64 up to 8192 (so the channel splits vary);
    sized for an oracle of about a second each."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n_cases:
        n = int(rng.integers(1, 10))
        Q = int(rng.integers(1, 17))
        d = 64 * int(rng.integers(1, 129))
        T = int(rng.choice([int(rng.integers(1, 40)), int(rng.integers(100, 200)), int(rng.integers(290, 700))]))
        if n * T * d * Q > 400_000_000:
            continue
        cases.append((T, n, Q, d))
    return cases


@pytest.mark.parametrize("T,n,Q,d", _random_interblock_cases())
def test_interblock_random_shapes(A, T, n, Q, d):
    test_interblock_pass_matches_the_oracle(A, n, Q, torch.bfloat16, d, True, T=T)


@pytest.mark.parametrize("T,n,Q", [(16, 8, 12), (64, 6, 12), (160, 8, 12), (153, 3, 5), (310, 8, 16),
                                   (1, 4, 12), (16, 2, 1)])
def test_interblock_tail_split_by_query_groups(A, T, n, Q):
    """The tokens of the last, partial round of the persistent grid are
    split by query groups over the idle CTAs: T = 16 (9 groups, 1-2 queries
    each), 64 (2 groups), 160 (8 leftover tokens, one query per CTA), 153
    (one leftover token, Q = 5 groups), 310 (6 leftover tokens, 16 groups),
    one token (12 CTAs, a query each), one query (no split)."""
    test_interblock_pass_matches_the_oracle(A, n, Q, torch.bfloat16, 7168, True, T=T)


@pytest.mark.parametrize("L,B,T,d,dtype", [
    (7, 3, 6, 64, torch.bfloat16),
    (9, 4, 7, 7168, torch.bfloat16),
    (93, 12, 16, 3584, torch.float32),     # the K3 layout at the fp32 bars
])
def test_two_phase_stack_matches_the_oracle(A, L, B, T, d, dtype):
    stk = W.stack(T=T, d=d, num_layers=L, block_size=B, seed=71 + L, device="cuda", dtype=dtype)
    fwd = _gpu_stack(A, stk, schedule="two_phase")
    store = O.round_bf16 if dtype == torch.bfloat16 else O.round_fp32
    tr = _oracle_stack(stk, store=store)
    tol = A_ATOL if dtype == torch.float32 else STACK_BF16_A_ATOL
    wa, wr = _check_stack(fwd, tr, slice(None), dtype, tol, check_blocks=(L < 20 or dtype == torch.float32))
    print(f"two-phase stack L={L} B={B} d={d} {dtype}: worst weight error {wa:.3g}, output {wr:.3g} x bound")


@pytest.mark.parametrize("L,B,T,d,dtype,start", [
    (93, 12, 16, 3584, torch.float32, 5),   # K3 layout: blocks 1-4 single pass, 5-8 two-phase
    (93, 12, 16, 7168, torch.bfloat16, 6),  # the default: blocks 6-8 two-phase (tensor-core logits, ring merge)
    (9, 2, 5, 7168, torch.bfloat16, 3),
    (7, 3, 6, 64, torch.float32, 9),        # start past the last block: all single pass
])
def test_hybrid_stack_matches_the_oracle(A, L, B, T, d, dtype, start):
    stk = W.stack(T=T, d=d, num_layers=L, block_size=B, seed=73 + L, device="cuda", dtype=dtype)
    fwd = _gpu_stack(A, stk, schedule="hybrid", two_phase_from=start)
    N = -(-L // B)
    # per two-phase block: the pass (two kernels with the tensor-core logits,
    # else one) and the step closing the block before, less the first
    # layer's merge, which the pass makes unnecessary
    per_pass = 2 if fwd.inter_ws is not None else 1
    assert fwd.launches_per_forward() == 2 * L + 1 + per_pass * max(0, N - start + 1)
    store = O.round_bf16 if dtype == torch.bfloat16 else O.round_fp32
    tr = _oracle_stack(stk, store=store)
    tol = A_ATOL if dtype == torch.float32 else STACK_BF16_A_ATOL
    wa, wr = _check_stack(fwd, tr, slice(None), dtype, tol, check_blocks=(L < 20 or dtype == torch.float32))
    print(f"hybrid stack L={L} B={B} from block {start}: worst weight error {wa:.3g}, output {wr:.3g} x bound")


def test_hybrid_graph_equals_eager(A):
    stk = W.stack(T=64, num_layers=93, block_size=12, seed=74, device="cuda")
    eager = _gpu_stack(A, stk, schedule="hybrid")
    graphed = _gpu_stack(A, stk, graph=True, schedule="hybrid")
    assert torch.equal(eager.r, graphed.r)
    for a1, a2 in zip(eager.weights, graphed.weights):
        assert torch.equal(a1, a2)


def test_two_phase_decode_T64_graph(A):
    stk = W.stack_T64(device="cuda")
    fwd = _gpu_stack(A, stk, graph=True, schedule="two_phase")
    tr = _oracle_stack(stk)
    wa, wr = _check_stack(fwd, tr, slice(None), torch.bfloat16, STACK_BF16_A_ATOL, check_blocks=False)
    print(f"two-phase decode stack T=64: worst weight error {wa:.3g}, output {wr:.3g} x bound")


def _random_stacks(n=10, seed=93):
    # seeded stack layouts: L 1..30, block size 1..12 (Full AttnRes to
    # one block), T 1..20, widths on the ring and the plain-load paths
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        L = int(rng.integers(1, 31))
        B = int(rng.integers(1, 13))
        T = int(rng.integers(1, 21))
        d = int(rng.choice([16, 64, 100, 256, 1000, 3584]))
        out.append((L, B, T, d, [torch.bfloat16, torch.float32][int(rng.integers(2))]))
    return out


@pytest.mark.parametrize("L,B,T,d,dtype", _random_stacks())
def test_random_stacks_against_oracle(A, L, B, T, d, dtype):
    stk = W.stack(T=T, d=d, num_layers=L, block_size=B, seed=7 * L + B + T, device="cuda", dtype=dtype)
    fwd = _gpu_stack(A, stk)
    store = O.round_bf16 if dtype == torch.bfloat16 else O.round_fp32
    tr = _oracle_stack(stk, store=store)
    tol = A_ATOL if dtype == torch.float32 else STACK_BF16_A_ATOL
    _check_stack(fwd, tr, slice(None), dtype, tol, check_blocks=dtype == torch.float32 or L <= 12)


def _random_two_phase_stacks(n=10, seed=2026):
    # seeded layouts for the two-phase and hybrid schedules: L 1..40, block
    # size 1..12, T 1..300 (the pass's query-split last round included),
    # widths the two-phase kernels take (tensor-core logits for bf16 with d
    # a multiple of 64, the CUDA-core pass otherwise), a random first
    # two-phase block
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        L = int(rng.integers(1, 41))
        B = int(rng.integers(1, 13))
        T = int(rng.integers(1, 301))
        dtype = [torch.bfloat16, torch.float32][int(rng.integers(2))]
        d = int(rng.choice([64, 256, 1000, 1024, 3584] + ([7168] if dtype == torch.bfloat16 else [])))
        if dtype == torch.float32 and d == 1000:
            continue
        N = -(-L // B)
        schedule = ["two_phase", "hybrid"][int(rng.integers(2))]
        start = int(rng.integers(1, N + 1))
        if T * d * L > 60_000_000:
            continue
        out.append((L, B, T, d, dtype, schedule, start))
    return out


@pytest.mark.parametrize("L,B,T,d,dtype,schedule,start", _random_two_phase_stacks())
def test_random_two_phase_stacks_against_oracle(A, L, B, T, d, dtype, schedule, start):
    stk = W.stack(T=T, d=d, num_layers=L, block_size=B, seed=11 * L + B + T, device="cuda", dtype=dtype)
    fwd = _gpu_stack(A, stk, schedule=schedule, two_phase_from=start)
    store = O.round_bf16 if dtype == torch.bfloat16 else O.round_fp32
    tr = _oracle_stack(stk, store=store)
    tol = A_ATOL if dtype == torch.float32 else STACK_BF16_A_ATOL
    _check_stack(fwd, tr, slice(None), dtype, tol, check_blocks=dtype == torch.float32 or L <= 12)
