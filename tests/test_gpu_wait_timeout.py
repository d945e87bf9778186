"""The timeout path of the bounded waits, exercised on a healthy GPU.

attnres_debug_wait_test(limit, row) makes every CTA's producer arm one row
of its first token without issuing its copy, and limits the main-loop
waits: the consumers' wait on that row runs out.  The kernel must then set
ATTNRES_DEVERR_WAIT_TIMEOUT, write NaN for the token it abandons, leave the
timed-out slot unreleased (no copy is ever issued into it again), stop its
producer, drain every copy it did issue, and return; after (0, -1) restores
normal operation the same call must give correct results.  Nothing here
faults or hangs a GPU: every wait is bounded and every issued copy targets
valid memory and is waited for before the CTA exits.
"""
import os
import subprocess
import sys

import pytest
import torch

import workloads as W
from tests.parity import check_weights, oracle_aggregate, to64

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000   # 1 ms: far above any healthy copy's latency
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# the opt-in cluster-split variant for few tokens (read once per process)
SPLIT = os.environ.get("ATTNRES_SPLIT", "0") not in ("", "0")


@pytest.fixture(scope="module")
def A():
    import depth_wise_attention_block_gb300 as A
    return A


@pytest.fixture(scope="module")
def TIMEOUT_BIT(A):
    return A.ATTNRES_DEVERR_WAIT_TIMEOUT


@pytest.fixture
def withheld(A):
    A.attnres_debug_wait_test(LIMIT_NS, 0)
    try:
        yield
    finally:
        A.attnres_debug_wait_test(0, -1)


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def test_aggregate_times_out_and_recovers(A, TIMEOUT_BIT):
    inp = W.block_T4096_d7168(device="cuda")
    r = torch.zeros((4096, 7168), dtype=torch.bfloat16, device="cuda")
    a = torch.zeros((4096, 9), device="cuda")
    err = _err()
    A.attnres_debug_wait_test(LIMIT_NS, 0)
    try:
        A.attnres_aggregate(inp.H, inp.w, r, a, dev_err=err)
        torch.cuda.synchronize()
    finally:
        A.attnres_debug_wait_test(0, -1)
    assert int(err.item()) & TIMEOUT_BIT
    # one CTA per SM; each abandons its first token (NaN) and writes nothing after it
    n = torch.cuda.get_device_properties(0).multi_processor_count
    assert torch.isnan(r[:n].float()).all() and torch.isnan(a[:n]).all()
    assert (r[n:] == 0).all() and (a[n:] == 0).all()
    # normal operation again: no error, correct weights
    err2 = _err()
    A.attnres_aggregate(inp.H, inp.w, r, a, dev_err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    idx = torch.arange(0, 4096, 97, device="cuda")
    _, a_ref, _, _ = oracle_aggregate(inp.H[:, idx].contiguous(), inp.w, 1e-5)
    check_weights(to64(a[idx]), a_ref)


def test_multi_group_times_out(A, TIMEOUT_BIT, withheld):
    inp = W.block_bf16(T=600, d=7168, seed=3, device="cuda", num_blocks=10)
    H = inp.H[:12].contiguous()
    r = torch.zeros((600, 7168), dtype=torch.bfloat16, device="cuda")
    err = _err()
    A.attnres_aggregate(H, inp.w, r, None, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & TIMEOUT_BIT
    assert torch.isnan(r[0].float()).all()


@pytest.mark.parametrize("prev", [False, True])
def test_multi_group_fold_times_out(A, TIMEOUT_BIT, withheld, prev):
    # a fused step over more than 9 sources: the multi-group kernel's fused
    # form, whose last group forms round(prev + F) (or takes F) and skips
    # its padding
    inp = W.block_bf16(T=600, d=7168, seed=3, device="cuda", num_blocks=10)
    stored = [inp.H[s] for s in range(11)]
    F = inp.H[11].clone()
    P = torch.zeros_like(F) if prev else None
    dst = torch.zeros_like(F)
    r = torch.zeros_like(F)
    err = _err()
    A.attnres_aggregate_fold(stored, P, F, dst, inp.w, r, None, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & TIMEOUT_BIT
    assert torch.isnan(r[0].float()).all()


def test_fused_stack_times_out(A, TIMEOUT_BIT, withheld):
    from depth_wise_attention_block_gb300.stack import StackForward
    stk = W.stack(T=256, num_layers=14, block_size=12, seed=9, device="cuda")
    err = _err()
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, 14, 12, dev_err=err, keep_weights=False)
    fwd.run()
    torch.cuda.synchronize()
    assert int(err.item()) & TIMEOUT_BIT


@pytest.mark.parametrize("schedule", ["two_phase", "hybrid"])
def test_two_phase_stack_times_out_and_recovers(A, TIMEOUT_BIT, schedule):
    # the two-phase schedule's ring kernels (the softmax / weighted-sum pass
    # after the tensor-core logits, the ring merge) abandon the withheld
    # token with the error bit set; run again normally, the same stack is
    # correct (equal to the single-pass schedule's weights to fp32 rounding)
    from depth_wise_attention_block_gb300.stack import StackForward
    stk = W.stack(T=256, num_layers=30, block_size=12, seed=10, device="cuda")
    err = _err()
    fwd = StackForward(stk.h0, stk.W, stk.G, stk.Sc, 30, 12, dev_err=err, schedule=schedule, two_phase_from=2)
    A.attnres_debug_wait_test(LIMIT_NS, 0)
    try:
        fwd.run()
        torch.cuda.synchronize()
    finally:
        A.attnres_debug_wait_test(0, -1)
    assert int(err.item()) & TIMEOUT_BIT
    err.zero_()
    fwd.run()
    ref = StackForward(stk.h0, stk.W, stk.G, stk.Sc, 30, 12)
    ref.run()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for a1, a2 in zip(fwd.weights, ref.weights):
        assert (a1 - a2).abs().max().item() <= 2e-2   # bf16 storage: rounding flips compound (the free-running bar)


def test_interblock_times_out_and_recovers(A, TIMEOUT_BIT):
    # the inter-block pass of the two-phase schedule keeps a token's rows in
    # the ring until the token is done: the withheld row's wait runs out,
    # the token's outputs for every query are NaN, nothing after it is
    # written, and the next call is correct again
    from tests.parity import oracle_aggregate
    T, n, Q = 600, 8, 12
    inp = W.block_bf16(T=T, d=7168, seed=7, device="cuda", num_blocks=n - 2)
    H = inp.H[:n].contiguous()
    g = torch.Generator(device="cuda").manual_seed(8)
    Wq = torch.randn((Q, 7168), generator=g, device="cuda") / 7168 ** 0.5
    R = torch.zeros((Q, T, 7168), device="cuda")
    lse = torch.zeros((Q, T), device="cuda")
    Aw = torch.zeros((Q, T, n), device="cuda")
    err = _err()
    A.attnres_debug_wait_test(LIMIT_NS, 0)
    try:
        A.attnres_interblock(list(H.unbind(0)), Wq, R, lse, Aw, dev_err=err)
        torch.cuda.synchronize()
    finally:
        A.attnres_debug_wait_test(0, -1)
    assert int(err.item()) & TIMEOUT_BIT
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert torch.isnan(R[:, :sms]).all() and torch.isnan(lse[:, :sms]).all() and torch.isnan(Aw[:, :sms]).all()
    assert (R[:, sms:] == 0).all() and (lse[:, sms:] == 0).all()
    err2 = _err()
    A.attnres_interblock(list(H.unbind(0)), Wq, R, lse, Aw, dev_err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    idx = torch.arange(0, T, 37, device="cuda")
    for q in (0, Q - 1):
        _, a_ref, _, _ = oracle_aggregate(H[:, idx].contiguous(), Wq[q], 1e-5)
        check_weights(to64(Aw[q, idx]), a_ref)


def test_backward_times_out_and_recovers(A, TIMEOUT_BIT):
    inp = W.block_bf16(T=1024, d=7168, seed=4, device="cuda")
    dr = torch.randn((1024, 7168), device="cuda").to(torch.bfloat16)
    gH = torch.zeros_like(inp.H)
    gw = torch.zeros(7168, device="cuda")
    err = _err()
    A.attnres_debug_wait_test(LIMIT_NS, 0)
    try:
        A.attnres_aggregate_backward(inp.H, inp.w, dr, gH, gw, dev_err=err)
        torch.cuda.synchronize()
    finally:
        A.attnres_debug_wait_test(0, -1)
    assert int(err.item()) & TIMEOUT_BIT
    err2 = _err()
    A.attnres_aggregate_backward(inp.H, inp.w, dr, gH, gw, dev_err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0 and torch.isfinite(gw).all()


def test_wait_test_rejects_bad_rows(A):
    with pytest.raises(Exception):
        A.attnres_debug_wait_test(LIMIT_NS, 8)


def test_split_variant_times_out_and_recovers(A, TIMEOUT_BIT):
    # the cluster-split variant shares each token across a cluster of CTAs;
    # at T = 64, d = 7168, S = 9 it takes clusters of 2, one token each.
    # Every CTA withholds a row of its (only) token: every token is
    # abandoned (NaN in r and the weights), the error bit is set, and
    # normal operation afterwards gives the one-CTA-per-token results.
    if not SPLIT:
        pytest.skip("runs in the child process of the next test (ATTNRES_SPLIT=1)")
    from tests.test_gpu_aggregate import _kernel_names
    inp = W.block_bf16(T=64, d=7168, seed=6, device="cuda")
    r = torch.zeros((64, 7168), dtype=torch.bfloat16, device="cuda")
    a = torch.zeros((64, 9), device="cuda")
    err = _err()
    A.attnres_debug_wait_test(LIMIT_NS, 0)
    try:
        names = _kernel_names(lambda: A.attnres_aggregate(inp.H, inp.w, r, a, dev_err=err))
        torch.cuda.synchronize()
    finally:
        A.attnres_debug_wait_test(0, -1)
    if names:
        assert any("agg_split_kernel" in n for n in names), names
    assert int(err.item()) & TIMEOUT_BIT
    assert torch.isnan(r.float()).all() and torch.isnan(a).all()
    err2 = _err()
    A.attnres_aggregate(inp.H, inp.w, r, a, dev_err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    _, a_ref, _, _ = oracle_aggregate(inp.H, inp.w, 1e-5)
    check_weights(to64(a), a_ref)


def test_split_variant_timeout_in_a_child_process():
    if SPLIT:
        pytest.skip("this is the child")
    env = dict(os.environ, ATTNRES_SPLIT="1")
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                          "tests/test_gpu_wait_timeout.py::test_split_variant_times_out_and_recovers"],
                         env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-2000:]
    assert "1 passed" in res.stdout, res.stdout[-2000:]
