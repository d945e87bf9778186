"""GPU parity of attnres_aggregate against the fp64 oracle, through the C ABI.

Covers the two named single-layer workloads at full size (T=64/d=256/S=4
fp32; T=4096/d=7168/S=9 bf16, every token), the long-context workload
(T=131072, on all outlier tokens plus a random sample), and shapes that
span several tiles with ragged tails: ragged token counts per CTA, rows
whose 16-byte vectors do not fill the last pass, every kernel (bulk-copy
ring, its multi-group and cluster-split variants, plain-load generic),
every dtype pairing, S = 1..128, T = 0 and 1, unaligned pointers.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads as W
from tests.parity import check_r, check_weights, oracle_aggregate, to64

pytestmark = pytest.mark.gpu

EPS = 1e-5
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# the opt-in cluster-split variant for few tokens (read once per process)
SPLIT = os.environ.get("ATTNRES_SPLIT", "0") not in ("", "0")


@pytest.fixture(scope="module")
def lib():
    import depth_wise_attention_block_gb300 as A
    return A


def _run(lib, H, w, out_dtype=torch.bfloat16, eps=EPS, with_weights=True):
    S, T, d = H.shape
    r = torch.full((T, d), float("nan"), dtype=out_dtype, device=H.device)
    a = torch.full((T, S), float("nan"), dtype=torch.float32, device=H.device) if with_weights else None
    err = torch.zeros(1, dtype=torch.int32, device=H.device)
    lib.attnres_aggregate(H, w, r, a, eps=eps, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return r, a


def _compare(H, w, r, a, out_dtype, eps=EPS):
    r_ref, a_ref, cond, M = oracle_aggregate(H, w, eps)
    if a is not None:
        check_weights(to64(a), a_ref)
    return check_r(to64(r), r_ref, out_dtype, cond, M)


def test_full_fp32_T64_d256_S4(lib):
    inp = W.full_T64_d256()
    H, w = inp.H.cuda(), inp.w.cuda()
    r, a = _run(lib, H, w, torch.float32)
    stats = _compare(H, w, r, a, torch.float32)
    print("full fp32 T64 d256:", stats)


def test_worked_example_four_sources_on_the_gpu(lib, golden_dir):
    # "Kimi K3 deep-dive (2)", section 2.1: weights [0.05, 0.10, 0.70, 0.15]
    # over h_0..h_3 give r_4 = 0.05 h_0 + 0.10 h_1 + 0.70 h_2 + 0.15 h_3.
    # Sources built (fp64, rounded to fp32) so their RMSNorm logits are
    # ln(a_s); the fp32 path must reproduce the page's weights within 1e-5
    # and its weighted sum within the fp32 bar.
    import math
    from tests.conftest import read_golden
    from tests.test_oracle_pins import _sources_with_logits
    rows = read_golden(os.path.join(golden_dir, "worked_example_4src.txt"))
    a_page = np.array([float(r[1]) for r in rows])
    d, T = 256, 7
    rng = np.random.default_rng(2024)
    w = (rng.standard_normal(d) / math.sqrt(d)).astype(np.float32).astype(np.float64)
    H = _sources_with_logits(w, np.log(a_page), d, T=T, rng=rng).astype(np.float32)
    Hg = torch.from_numpy(H).cuda()
    r, a = _run(lib, Hg, torch.from_numpy(w.astype(np.float32)).cuda(), torch.float32)
    assert np.abs(to64(a) - a_page[None]).max() <= 1e-5
    H64 = H.astype(np.float64)
    r_page = np.einsum("s,std->td", a_page, H64)
    cond = np.einsum("s,std->td", a_page, np.abs(H64))
    assert (np.abs(to64(r) - r_page) <= 1e-5 * (np.abs(r_page) + cond)).all()


def test_block_bf16_T4096_d7168_S9_every_token(lib):
    inp = W.block_T4096_d7168(device="cuda")
    r, a = _run(lib, inp.H, inp.w, torch.bfloat16)
    stats = _compare(inp.H, inp.w, r, a, torch.bfloat16)
    print("block bf16 T4096 d7168:", stats)
    assert torch.allclose(a.sum(1), torch.ones(4096, device="cuda"), atol=1e-6)


def test_long_context_T131072_sampled(lib):
    inp = W.block_T131072_d7168(device="cuda")
    r, a = _run(lib, inp.H, inp.w, torch.bfloat16)
    g = torch.Generator().manual_seed(99)
    rnd = torch.randperm(131072, generator=g)[:8192].to("cuda")
    idx = torch.unique(torch.cat([inp.outlier_tokens, rnd]))
    assert inp.outlier_tokens.numel() == 1311
    Hs = inp.H[:, idx].contiguous()
    stats = _compare(Hs, inp.w, r[idx], a[idx], torch.bfloat16)
    print(f"long context: {idx.numel()} tokens checked:", stats)
    # a x50 source keeps its RMSNorm'd logit: the weights stay finite, no NaN
    assert torch.isfinite(r).all() and torch.isfinite(a).all()


# (T, d, S, src dtype, out dtype) -- comments say which kernel and why
SHAPES = [
    (1000, 7168, 9, torch.bfloat16, torch.bfloat16),   # ring, 2 vectors/thread, ragged T over CTAs
    (333, 7160, 9, torch.bfloat16, torch.bfloat16),    # ring, 895 vectors: ragged last pass
    (257, 3592, 5, torch.bfloat16, torch.float32),     # ring, 449 vectors, fp32 out
    (77, 3584, 9, torch.bfloat16, torch.bfloat16),     # ring, exactly 448 vectors
    (129, 1000, 7, torch.float32, torch.bfloat16),     # ring, fp32 in, bf16 out (8-byte stores)
    (300, 3584, 9, torch.float32, torch.float32),      # ring, fp32, 2 vectors/thread
    (50, 7176, 9, torch.bfloat16, torch.bfloat16),     # generic: 897 vectors > 2 per thread
    (40, 7168, 12, torch.bfloat16, torch.bfloat16),    # multi-group ring: S > 9 (groups of 6)
    (300, 7168, 94, torch.bfloat16, torch.bfloat16),   # multi-group ring: Full AttnRes top layer, 94 sources
    (200, 3584, 17, torch.float32, torch.float32),     # multi-group ring, fp32 (groups of 9)
    (129, 7160, 10, torch.bfloat16, torch.float32),    # multi-group ring, ragged last vector pass
    (50, 1000, 128, torch.float32, torch.bfloat16),    # multi-group ring, S = 128, one vector per thread
    (31, 7, 3, torch.float32, torch.float32),          # generic: row not a 16-byte multiple
    (31, 100, 128, torch.bfloat16, torch.float32),     # generic: S = 128
    (3, 7168, 1, torch.bfloat16, torch.bfloat16),      # S = 1
    (1, 7168, 9, torch.bfloat16, torch.bfloat16),      # T = 1
    (5, 64, 2, torch.bfloat16, torch.bfloat16),        # tiny row: 8 vectors
    (7, 8, 9, torch.bfloat16, torch.bfloat16),         # ring, one 16-byte vector per row
    (13, 1, 4, torch.float32, torch.float32),          # d = 1: one channel (generic)
    (9, 1, 9, torch.bfloat16, torch.bfloat16),         # d = 1, bf16 (generic)
    # few tokens: a cluster of C CTAs per token, each a channel slice
    (64, 7168, 9, torch.bfloat16, torch.bfloat16),     # split C=2, 448 vectors per CTA (decode size)
    (19, 7168, 9, torch.bfloat16, torch.bfloat16),     # split C=8, 112 vectors: partial last warp
    (38, 7168, 5, torch.float32, torch.float32),       # split C=4, fp32
    (17, 4096, 9, torch.float32, torch.bfloat16),      # split C=8, fp32 in, bf16 out (8-byte stores)
    (70, 2048, 7, torch.bfloat16, torch.float32),      # split C=2, 128 vectors, fp32 out
    (76, 1024, 9, torch.bfloat16, torch.bfloat16),     # split C=2, 64 vectors, C*T = 152 exactly
    (2, 7168, 2, torch.bfloat16, torch.bfloat16),      # split C=8, S = 2
]


@pytest.mark.parametrize("T,d,S,sdt,odt", SHAPES)
def test_shapes(lib, T, d, S, sdt, odt):
    inp = W.block_bf16(T=T, d=d, seed=1000 + T + d + S, device="cuda", num_blocks=max(S - 2, 0),
                       src_dtype=sdt)
    H = inp.H[:S].contiguous()
    r, a = _run(lib, H, inp.w, odt)
    _compare(H, inp.w, r, a, odt)
    if S == 1:
        assert torch.equal(r.float(), H[0].float()) and torch.equal(a, torch.ones_like(a))


def test_rows_beyond_2_gib_use_64_bit_offsets(lib):
    # T = 160000 bf16 rows of d = 7168: a source spans 2.29 GB, so the later
    # tokens' rows start beyond 2^31 bytes (64-bit offsets in every kernel
    # address); the last tokens are checked against the oracle
    T, d = 160000, 7168
    g = torch.Generator(device="cuda").manual_seed(17)
    H = torch.empty((2, T, d), dtype=torch.bfloat16, device="cuda")
    for s in range(2):
        H[s].normal_(generator=g).mul_(1.0 + s)
    w = torch.randn(d, generator=g, device="cuda") / d ** 0.5
    r, a = _run(lib, H, w, torch.bfloat16)
    tail = torch.arange(T - 300, T, device="cuda")
    _compare(H[:, tail].contiguous(), w, r[tail], a[tail], torch.bfloat16)
    del H, r, a
    torch.cuda.empty_cache()


def test_split_matches_one_cta_per_token(lib):
    # the first 64 tokens alone take the cluster kernel, all 4096 the
    # one-CTA-per-token ring: same values up to the order of fp32 sums
    inp = W.block_T4096_d7168(device="cuda")
    r_ring, a_ring = _run(lib, inp.H, inp.w, torch.float32)
    H64 = inp.H[:, :64].contiguous()
    r_split, a_split = _run(lib, H64, inp.w, torch.float32)
    assert (a_split - a_ring[:64]).abs().max().item() < 5e-6
    scale = inp.H[:, :64].float().abs().amax(0)
    # |a_s| differ by < 5e-6 each over 9 sources, plus fp32 rounding of r
    assert ((r_split - r_ring[:64]).abs() <= 6e-5 * scale + 1e-30).all()


def _kernel_names(fn):
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    return [e.name for e in prof.events() if "agg_" in e.name]


def test_dispatch_picks_the_expected_kernel(lib):
    inp = W.block_bf16(T=4096, d=7168, seed=3, device="cuda")
    cases = [  # (sources, tokens, expected kernel)
        (inp.H, 4096, "agg_ring_kernel"),
        (inp.H[:, :64].contiguous(), 64, "agg_split_kernel" if SPLIT else "agg_ring_kernel"),
        (inp.H[:, :64, :7160].contiguous(), 64, "agg_ring_kernel"),  # 895 vectors: no even split
        (torch.cat([inp.H[:, :40]] * 2)[:12].contiguous(), 40, "agg_ring_multi_kernel"),
    ]
    seen_any = False
    for H, T, want in cases:
        r = torch.empty((T, H.shape[2]), dtype=torch.bfloat16, device="cuda")
        names = _kernel_names(lambda: lib.attnres_aggregate(H, inp.w[: H.shape[2]], r))
        if not names:
            continue
        seen_any = True
        assert len(names) == 1 and names[0].split("<")[0].split("(")[0].split()[-1].endswith(want), (want, names)
    if not seen_any:
        pytest.skip("the profiler recorded no kernels")


def test_split_variant_parity_in_a_child_process():
    # the cluster-split variant is opt-in per process: run the few-token
    # parity tests again in a child with it switched on
    if SPLIT:
        pytest.skip("this is the child")
    env = dict(os.environ, ATTNRES_SPLIT="1")
    tests = ["tests/test_gpu_aggregate.py::test_shapes",
             "tests/test_gpu_aggregate.py::test_split_matches_one_cta_per_token",
             "tests/test_gpu_aggregate.py::test_dispatch_picks_the_expected_kernel",
             "tests/test_gpu_stack.py::test_fused_equals_unfused_bit_for_bit",
             "tests/test_gpu_stack.py::test_decode_stack_T64_every_token",
             "tests/test_gpu_stack.py::test_full_attnres_fp32_storage_93_layers"]
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"] + tests,
                         env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-2000:]
    print(res.stdout.strip().splitlines()[-1])


def test_unaligned_pointers_take_the_generic_path(lib):
    T, d, S = 64, 7168, 9
    inp = W.block_bf16(T=T, d=d, seed=5, device="cuda")
    big = torch.empty(S * T * d + 1, dtype=torch.bfloat16, device="cuda")
    H = big[1:].view(S, T, d)          # 2-byte offset: not 16-byte aligned
    H.copy_(inp.H)
    r, a = _run(lib, H, inp.w)
    _compare(H, inp.w, r, a, torch.bfloat16)
    r2, a2 = _run(lib, inp.H, inp.w)
    # same values from the other kernel, within a few fp32 ulps
    assert (a - a2).abs().max().item() < 5e-6


def test_empty_T_writes_nothing(lib):
    H = torch.zeros((3, 0, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, device="cuda")
    r = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    lib.attnres_aggregate(H, w, r)
    torch.cuda.synchronize()


def test_weights_optional(lib):
    inp = W.block_bf16(T=200, d=7168, seed=6, device="cuda")
    r1, _ = _run(lib, inp.H, inp.w, with_weights=False)
    r2, _ = _run(lib, inp.H, inp.w, with_weights=True)
    assert torch.equal(r1, r2)


def test_zero_query_gives_the_mean(lib):
    inp = W.block_bf16(T=100, d=7168, seed=7, device="cuda", src_dtype=torch.float32)
    w = torch.zeros_like(inp.w)
    r, a = _run(lib, inp.H, w, torch.float32)
    assert torch.allclose(a, torch.full_like(a, 1 / 9), atol=1e-7)
    _compare(inp.H, w, r, a, torch.float32)


def test_deterministic_across_runs(lib):
    inp = W.block_bf16(T=512, d=7168, seed=8, device="cuda")
    r1, a1 = _run(lib, inp.H, inp.w)
    r2, a2 = _run(lib, inp.H, inp.w)
    assert torch.equal(r1, r2) and torch.equal(a1, a2)


def _host_copy(t: torch.Tensor, pinned: bool) -> torch.Tensor:
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=pinned)
    h.copy_(t)
    return h


@pytest.mark.parametrize("chunk,slots", [(1000, 1), (256, 2), (333, 3), (256, 1), (7, 2)])
def test_aggregate_host_matches_device_path(lib, chunk, slots):
    # host buffers in and out through the C ABI, chunked over tokens through
    # a ring of staging slots: every token is computed by the same arithmetic
    # as in one launch over all tokens, so bit for bit
    T, d, S = 1000, 7168, 9
    inp = W.block_bf16(T=T, d=d, seed=9, device="cuda")
    H_host, w_host = _host_copy(inp.H, True), _host_copy(inp.w, True)
    r_host = torch.full((T, d), float("nan"), dtype=torch.bfloat16, pin_memory=True)
    a_host = torch.full((T, S), float("nan"), dtype=torch.float32, pin_memory=True)
    nbytes = lib.attnres_aggregate_host_workspace_size(S, min(chunk, T), d, torch.bfloat16, torch.bfloat16, True, slots)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r_ref, a_ref = _run(lib, inp.H, inp.w)
    for _ in range(2):  # a second call reuses the slots with stale contents
        lib.attnres_aggregate_host(H_host, w_host, r_host, a_host, workspace=ws, chunk_tokens=chunk, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(r_host.cuda(), r_ref) and torch.equal(a_host.cuda(), a_ref)
        r_host.fill_(float("nan"))
        a_host.fill_(float("nan"))


def test_aggregate_host_pageable_fp32_ragged_rows_against_oracle(lib):
    # pageable (not page-locked) host memory, fp32, rows of 100 channels (not
    # a whole number of 16-byte vectors: the plain-load kernel), a ragged last
    # chunk, no weights; checked against the oracle and the device path
    g = torch.Generator().manual_seed(31)
    S, T, d = 4, 37, 100
    H = torch.randn(S, T, d, generator=g) * torch.tensor([0.5, 1.0, 2.0, 4.0]).view(S, 1, 1)
    w = torch.randn(d, generator=g) / d ** 0.5
    r_host = torch.full((T, d), float("nan"), dtype=torch.float32)
    lib.attnres_aggregate_host(list(H.unbind(0)), w, r_host, None, chunk_tokens=5)
    torch.cuda.synchronize()
    assert not torch.isnan(r_host).any()
    _compare(H, w, r_host, None, torch.float32)
    r_dev, _ = _run(lib, H.cuda(), w.cuda(), torch.float32, with_weights=False)
    assert torch.equal(r_host, r_dev.cpu())


def test_aggregate_host_orders_after_stream_work(lib):
    # the call is ordered after work already queued on its stream (a long
    # kernel here), and an event recorded on the stream after the call
    # completes only once the host outputs are final
    S, T, d = 3, 64, 256
    g = torch.Generator().manual_seed(32)
    H = torch.randn(S, T, d, generator=g)
    w = torch.randn(d, generator=g) / 16
    stream = torch.cuda.Stream()
    r_host = torch.full((T, d), float("nan"), dtype=torch.float32, pin_memory=True)
    a_host = torch.full((T, S), float("nan"), dtype=torch.float32, pin_memory=True)
    H_host, w_host = _host_copy(H, True), _host_copy(w, True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)  # a long kernel ahead of the call on its stream
        lib.attnres_aggregate_host(H_host, w_host, r_host, a_host, chunk_tokens=16, stream=stream)
        done = torch.cuda.Event()
        done.record(stream)
    done.synchronize()
    r_dev, a_dev = _run(lib, H.cuda(), w.cuda(), torch.float32)
    assert torch.equal(r_host, r_dev.cpu()) and torch.equal(a_host, a_dev.cpu())


def test_aggregate_host_refuses_a_capturing_stream(lib):
    # its copy streams cannot join a graph capture: the call is refused
    # before it enqueues anything, and the capture itself stays valid
    S, T, d = 2, 16, 256
    H_host = torch.randn(S, T, d).pin_memory()
    w_host = torch.randn(d).pin_memory()
    r_host = torch.empty((T, d), dtype=torch.float32, pin_memory=True)
    nbytes = lib.attnres_aggregate_host_workspace_size(S, 8, d, torch.float32, torch.float32, False, 2)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with pytest.raises(lib.AttnresError, match="captured"):
        with torch.cuda.graph(graph, stream=side):
            lib.attnres_aggregate_host(H_host, w_host, r_host, None, workspace=ws, chunk_tokens=8, stream=side)
    torch.cuda.synchronize()


def test_stacked_list_and_strided_sources_agree(lib):
    # the binding takes a contiguous [S, T, d] stack by pointer arithmetic, a
    # list one tensor at a time, and a strided stack (every other source of a
    # larger one) slice by slice: the same sources give the same bits
    inp = W.block_bf16(T=200, d=7168, seed=12, device="cuda")
    S, T, d = inp.H.shape
    r1, a1 = _run(lib, inp.H, inp.w)
    r2 = torch.empty_like(r1)
    a2 = torch.empty_like(a1)
    lib.attnres_aggregate(list(inp.H.unbind(0)), inp.w, r2, a2)
    wide = torch.zeros((2 * S, T, d), dtype=inp.H.dtype, device="cuda")
    wide[::2] = inp.H
    r3 = torch.empty_like(r1)
    a3 = torch.empty_like(a1)
    lib.attnres_aggregate(wide[::2], inp.w, r3, a3)
    torch.cuda.synchronize()
    assert torch.equal(r1, r2) and torch.equal(a1, a2)
    assert torch.equal(r1, r3) and torch.equal(a1, a3)
    with pytest.raises(ValueError):
        lib.attnres_aggregate(inp.H[:0], inp.w, r1, None)


def test_aggregate_host_multi_group_fp32_out(lib):
    # more than 9 sources (the multi-group kernel) through the host-buffer
    # call, fp32 output, a ragged last chunk: bit for bit the device path
    T, d, S = 50, 7168, 20
    inp = W.full_bf16(T=T, d=d, S=S, seed=13, device="cuda")
    H_host, w_host = _host_copy(inp.H, True), _host_copy(inp.w, True)
    r_host = torch.full((T, d), float("nan"), dtype=torch.float32, pin_memory=True)
    a_host = torch.full((T, S), float("nan"), dtype=torch.float32, pin_memory=True)
    lib.attnres_aggregate_host(H_host, w_host, r_host, a_host, chunk_tokens=16)
    torch.cuda.synchronize()
    r_ref, a_ref = _run(lib, inp.H, inp.w, torch.float32)
    assert torch.equal(r_host.cuda(), r_ref) and torch.equal(a_host.cuda(), a_ref)
    _compare(inp.H, inp.w, r_host, a_host, torch.float32)


def _random_cases(n=32, seed=2026):
    # seeded shapes over every dispatch path: T 1..400, d 1..8192 (row
    # lengths that are and are not whole 16-byte vectors), S 1..128, all
    # dtype pairings; sized so the oracle finishes each in about a second
    rng = np.random.default_rng(seed)
    dts = [torch.bfloat16, torch.float32]
    cases = []
    while len(cases) < n:
        S = int(rng.choice([1, 2, 3, 5, 8, 9, 10, 13, 24, 47, 94, 128]))
        d = int(rng.choice([1, 7, 8, 64, 100, 256, 1000, 3584, 3592, 7160, 7168, 8192]))
        T = int(rng.integers(1, 401))
        if S * T * d > 12_000_000:
            continue
        cases.append((T, d, S, dts[int(rng.integers(2))], dts[int(rng.integers(2))]))
    return cases


@pytest.mark.parametrize("T,d,S,sdt,odt", _random_cases())
def test_random_shapes_against_oracle(lib, T, d, S, sdt, odt):
    g = torch.Generator(device="cuda").manual_seed(T * 131 + d * 7 + S)
    sig = torch.exp(torch.randn(S, 1, 1, generator=g, device="cuda"))  # a scale per source
    H = (torch.randn(S, T, d, generator=g, device="cuda") * sig).to(sdt)
    w = torch.randn(d, generator=g, device="cuda") / max(d, 1) ** 0.5
    r, a = _run(lib, H, w, odt)
    _compare(H, w, r, a, odt)
