"""GPU parity of attnres_aggregate_backward (gradients with respect to the
sources and the pseudo-query, forward recomputed) against the fp64 oracle.

Bars: fp32 gradients within 1e-5 of their condition scale (the same sums
over absolute values, from the oracle); bf16 gradients within one bf16 ulp
plus 1e-3 of the token's largest condition scale; grad_w (fp32) within 1e-5
of its condition scale.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.parity import oracle_backward, to64, ulp_bf16

pytestmark = pytest.mark.gpu
EPS = 1e-5


@pytest.fixture(scope="module")
def A():
    import depth_wise_attention_block_gb300 as A
    return A


def _inputs(T, d, S, dtype, seed):
    inp = W.block_bf16(T=T, d=d, seed=seed, device="cuda", num_blocks=max(S - 2, 0), src_dtype=dtype)
    H = inp.H[:S].contiguous()
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    dr = torch.randn((T, d), generator=g, device="cuda").to(dtype)
    return H, inp.w, dr


def _run(A, H, w, dr, accumulate=False, init=None):
    S, T, d = H.shape
    gH = torch.zeros_like(H) if init is None else init.clone()
    gw = torch.full((d,), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    A.attnres_aggregate_backward(H, w, dr, gH, gw, eps=EPS, accumulate=accumulate, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return gH, gw


def _check(gH, gw, dH, dw, dHs, dws, dtype):
    e_w = np.abs(to64(gw) - dw)
    assert (e_w <= 1e-5 * dws + 1e-30).all(), f"grad_w: worst {np.max(e_w / (dws + 1e-30)):.3g} x scale"
    e_h = np.abs(to64(gH) - dH)
    if dtype == torch.float32:
        bound = 1e-5 * dHs
    else:
        bound = ulp_bf16(dH) + 1e-3 * dHs.max(axis=2, keepdims=True)
    ratio = e_h / np.maximum(bound, 1e-300)
    assert (e_h <= bound).all(), f"grad sources: worst {ratio.max():.3g} x bound"
    return float(ratio.max())


SHAPES = [
    (4096, 7168, 9, torch.bfloat16),   # ring, K3 width
    (300, 3584, 9, torch.float32),     # ring, fp32, 2 vectors/thread
    (333, 7160, 5, torch.bfloat16),    # ring, ragged vectors
    (129, 1000, 3, torch.float32),     # ring, 1 vector/thread
    (50, 7168, 1, torch.bfloat16),     # one source: grad = dr, grad_w = 0
    (40, 3584, 12, torch.float32),     # generic: S > 9
    (31, 100, 7, torch.float32),       # generic: row not a 16-byte multiple
]


@pytest.mark.parametrize("T,d,S,dtype", SHAPES)
def test_backward_parity(A, T, d, S, dtype):
    H, w, dr = _inputs(T, d, S, dtype, seed=T + d + S)
    gH, gw = _run(A, H, w, dr)
    dH, dw, dHs, dws = oracle_backward(H, w, dr, EPS)
    worst = _check(gH, gw, dH, dw, dHs, dws, dtype)
    print(f"backward T={T} d={d} S={S} {dtype}: worst {worst:.3g} x bound")
    if S == 1:
        assert torch.equal(gH[0], dr) and torch.count_nonzero(gw) == 0


def test_backward_accumulates(A):
    H, w, dr = _inputs(200, 7168, 9, torch.float32, seed=3)
    g = torch.Generator(device="cuda").manual_seed(4)
    init = torch.randn(H.shape, generator=g, device="cuda")
    _, gw1 = _run(A, H, w, dr)
    acc, gw2 = _run(A, H, w, dr, accumulate=True, init=init)
    dH, dw, dHs, dws = oracle_backward(H, w, dr, EPS)
    want = to64(init) + dH
    assert (np.abs(to64(acc) - want) <= 1e-5 * (dHs + np.abs(to64(init)))).all()
    assert torch.equal(gw1, gw2)


def test_backward_grad_w_is_reproducible(A):
    H, w, dr = _inputs(1000, 7168, 9, torch.bfloat16, seed=5)
    _, gw1 = _run(A, H, w, dr)
    _, gw2 = _run(A, H, w, dr)
    assert torch.equal(gw1, gw2)


def test_backward_empty_T_zeroes_grad_w(A):
    d = 64
    gw = torch.full((d,), 7.0, device="cuda")
    H = torch.zeros((2, 0, d), dtype=torch.float32, device="cuda")
    A.attnres_aggregate_backward(H, torch.zeros(d, device="cuda"), torch.zeros((0, d), device="cuda"),
                                 torch.zeros_like(H), gw, workspace=torch.zeros(1, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(gw) == 0


def _random_cases(n=20, seed=77):
    # seeded shapes for the backward: T 1..300, d from 8 to 8192, S 1..24
    # (the ring backward up to 9 sources, the plain-load one beyond and for
    # rows that are not whole 16-byte vectors), both dtypes, accumulate or
    # not; small enough for the oracle backward to take about a second
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        S = int(rng.choice([1, 2, 3, 5, 8, 9, 12, 24]))
        d = int(rng.choice([8, 64, 100, 1000, 3584, 3592, 7160, 7168, 8192]))
        T = int(rng.integers(1, 301))
        if S * T * d > 6_000_000:
            continue
        dtype = [torch.bfloat16, torch.float32][int(rng.integers(2))]
        cases.append((T, d, S, dtype, bool(rng.integers(2))))
    return cases


@pytest.mark.parametrize("T,d,S,dtype,acc", _random_cases())
def test_backward_random_shapes(A, T, d, S, dtype, acc):
    g = torch.Generator(device="cuda").manual_seed(T * 17 + d + S)
    sig = torch.exp(0.5 * torch.randn(S, 1, 1, generator=g, device="cuda"))
    H = (torch.randn(S, T, d, generator=g, device="cuda") * sig).to(dtype)
    w = torch.randn(d, generator=g, device="cuda") / d ** 0.5
    dr = torch.randn((T, d), generator=g, device="cuda").to(dtype)
    init = torch.randn(H.shape, generator=g, device="cuda").to(dtype) if acc else None
    gH, gw = _run(A, H, w, dr, accumulate=acc, init=init)
    dH, dw, dHs, dws = oracle_backward(H, w, dr, EPS)
    if acc:
        # the old gradients are added: the bar grows by their size
        dH = dH + to64(init)
        dHs = dHs + np.abs(to64(init))
    _check(gH, gw, dH, dw, dHs, dws, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_autograd_function_against_the_oracle(A, dtype):
    # aggregate(H, w) in a torch graph: its forward equals attnres_aggregate
    # bit for bit and the gradients of sum(r * dr) are the oracle's
    from depth_wise_attention_block_gb300.autograd import aggregate
    H0, w0, dr = _inputs(300, 3584, 9, dtype, seed=21)
    H = H0.clone().requires_grad_(True)
    w = w0.clone().requires_grad_(True)
    r = aggregate(H, w)
    r_ref = torch.empty_like(r)
    A.attnres_aggregate(H0, w0, r_ref)
    assert torch.equal(r.detach(), r_ref)
    (r.float() * dr.float()).sum().backward()
    dH, dw, dHs, dws = oracle_backward(H0, w0, dr, EPS)
    assert H.grad.dtype == dtype and w.grad.dtype == torch.float32
    _check(H.grad, w.grad, dH, dw, dHs, dws, dtype)
    # only the query learns: no source gradient is formed
    w2 = w0.clone().requires_grad_(True)
    (aggregate(H0, w2).float() * dr.float()).sum().backward()
    assert torch.equal(w2.grad, w.grad)
