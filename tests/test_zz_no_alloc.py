"""attnres_aggregate_backward_noalloc: the backward for callers that cannot
allocate device memory (a fixed memory budget, or no cudaMalloc once the
process is serving).  Its scratch workspace is an array built into the
library instead of a caller buffer.

Checked through the C ABI: two calls in a row (different shapes and dtypes,
so the second starts on the first one's leftover scratch) give the same
gradients as attnres_aggregate_backward with a caller workspace, within the
backward parity bar; a request larger than the built-in scratch is refused;
and a plain C client gets the same gradients before and after a
cudaDeviceReset.  This file is collected last so that a run stopping at the first failure
has run every other test before it.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import workloads as W
from tests.parity import oracle_backward, to64, ulp_bf16

pytestmark = pytest.mark.gpu
EPS = 1e-5


def _inputs(T, d, S, dtype, seed):
    inp = W.block_bf16(T=T, d=d, seed=seed, device="cuda", num_blocks=max(S - 2, 0), src_dtype=dtype)
    H = inp.H[:S].contiguous()
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    dr = torch.randn((T, d), generator=g, device="cuda").to(dtype)
    return H, inp.w, dr


def _call_noalloc(A, H, w, dr, gH, gw):
    S, T, d = H.shape
    sp = (ctypes.c_void_p * S)(*[H[s].data_ptr() for s in range(S)])
    gp = (ctypes.c_void_p * S)(*[gH[s].data_ptr() for s in range(S)])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = A._N.lib.attnres_aggregate_backward_noalloc(
        sp, S, T, d, A.dtype_code(H.dtype), w.data_ptr(), EPS, dr.data_ptr(), gp, 0, gw.data_ptr(),
        err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return rc, err


def test_noalloc_backward_matches_workspace_backward_twice():
    import depth_wise_attention_block_gb300 as A
    for T, d, S, dtype, seed in [(2048, 7168, 9, torch.bfloat16, 21), (700, 3584, 4, torch.float32, 22)]:
        H, w, dr = _inputs(T, d, S, dtype, seed)
        ref_gH = torch.empty_like(H)
        ref_gw = torch.empty(d, device="cuda")
        A.attnres_aggregate_backward(H, w, dr, ref_gH, ref_gw, eps=EPS)
        gH = torch.full_like(H, float("nan"))
        gw = torch.full((d,), float("nan"), device="cuda")
        rc, err = _call_noalloc(A, H, w, dr, gH, gw)
        torch.cuda.synchronize()
        assert rc == 0, A._N.lib.attnres_last_error()
        assert int(err.item()) == 0
        # the parity bar of the backward tests, around the workspace entry point's result
        _, _, dHs, dws = oracle_backward(H, w, dr, EPS)
        assert (np.abs(to64(gw) - to64(ref_gw)) <= 1e-5 * dws + 1e-30).all()
        ref = to64(ref_gH)
        bound = 1e-5 * dHs if dtype == torch.float32 else ulp_bf16(ref) + 1e-3 * dHs.max(axis=2, keepdims=True)
        assert (np.abs(to64(gH) - ref) <= bound).all()
        print(f"no-alloc backward T={T} d={d} S={S} {dtype}: bitwise equal = "
              f"{torch.equal(gH, ref_gH) and torch.equal(gw, ref_gw)}")


def test_noalloc_backward_refuses_oversize():
    import depth_wise_attention_block_gb300 as A
    # one fp32 row of d per CTA, min(T, SMs) CTAs: pick d just past the
    # built-in 1,310,720 values
    T, S = 200, 2
    rows = min(T, torch.cuda.get_device_properties(0).multi_processor_count)
    d = 8 * (1310720 // (8 * rows) + 1)
    H, w, dr = _inputs(T, d, S, torch.float32, 5)
    gH, gw = torch.zeros_like(H), torch.zeros(d, device="cuda")
    rc, _ = _call_noalloc(A, H, w, dr, gH, gw)
    assert rc == A._N.ATTNRES_ERANGE
    assert b"built-in scratch" in A._N.lib.attnres_last_error()


def test_noalloc_backward_survives_a_device_reset(tmp_path):
    # A caller that resets its device (cudaDeviceReset: a new context, the
    # library's module loaded again) must get the same gradients from the
    # no-alloc backward afterwards: the scratch array's address and the
    # kernels' shared-memory opt-in are looked up again for the new
    # context.  Run from a plain C client (tests/c_abi/noalloc_reset_client.c)
    # in a process of its own, so the reset touches nothing else.
    import __graft_entry__
    B = __graft_entry__._build_module()
    if not os.path.exists(B.LIB_PATH):
        B.build()
    lib = os.path.abspath(B.LIB_PATH)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    nv = shutil.which("nvcc")
    cuda = os.environ.get("CUDA_HOME") or (os.path.dirname(os.path.dirname(nv)) if nv else "/usr/local/cuda")
    exe = tmp_path / "noalloc_reset_client"
    build = subprocess.run(
        ["gcc", "-O2", "-std=c11", "-Wall", "-I", os.path.join(root, "include"), "-I", os.path.join(cuda, "include"),
         os.path.join(root, "tests", "c_abi", "noalloc_reset_client.c"), "-o", str(exe), lib,
         f"-L{cuda}/lib64", "-lcudart", f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{cuda}/lib64"],
        capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr + run.stdout
    assert "equal before and after cudaDeviceReset" in run.stdout
