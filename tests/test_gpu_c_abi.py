"""The C ABI from a plain C program, with no Python or torch in the caller:
tests/c_abi/abi_client.c is built with gcc against include/attnres.h,
libattnres.so and the CUDA runtime, and run on the GPU.  It checks on its
own that the host-buffer call agrees bit for bit with the device-buffer one
and that a bad argument is refused; its inputs and outputs are then checked
here against the fp64 oracle at the bf16 bars."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle as O
from tests.parity import check_r, check_weights

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home() -> str:
    nv = shutil.which("nvcc")
    if os.environ.get("CUDA_HOME"):
        return os.environ["CUDA_HOME"]
    return os.path.dirname(os.path.dirname(nv)) if nv else "/usr/local/cuda"


def _bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _build_and_run(tmp_path, name):
    """Build tests/c_abi/<name>.c with gcc against the library and run it;
    returns the bytes it wrote."""
    import __graft_entry__
    B = __graft_entry__._build_module()
    if not os.path.exists(B.LIB_PATH):
        B.build()
    lib = os.path.abspath(B.LIB_PATH)
    cuda = _cuda_home()
    exe = tmp_path / name
    build = subprocess.run(
        ["gcc", "-O2", "-std=c11", "-Wall", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
         os.path.join(ROOT, "tests", "c_abi", f"{name}.c"), "-o", str(exe), lib,
         f"-L{cuda}/lib64", "-lcudart", f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{cuda}/lib64"],
        capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    out = tmp_path / "out.bin"
    run = subprocess.run([str(exe), str(out)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr + run.stdout
    return out.read_bytes()


def test_c_client_against_the_oracle(tmp_path):
    raw = _build_and_run(tmp_path, "abi_client")

    S, T, d = (int(v) for v in np.frombuffer(raw[:12], dtype=np.int32))
    off = 12
    src = np.frombuffer(raw, np.uint16, S * T * d, off)
    off += S * T * d * 2
    w = np.frombuffer(raw, np.float32, d, off)
    off += d * 4
    r_bits = np.frombuffer(raw, np.uint16, T * d, off)
    off += T * d * 2
    a = np.frombuffer(raw, np.float32, T * S, off).reshape(T, S).astype(np.float64)
    assert off + T * S * 4 == len(raw)

    H = _bf16_bits_to_f64(src).reshape(S, T, d)
    r = _bf16_bits_to_f64(r_bits).reshape(T, d)
    r_ref, a_ref = O.depth_attention(H, w.astype(np.float64), 1e-5)
    check_weights(a, a_ref)
    M = np.abs(H).max(axis=(0, 2))
    stats = check_r(r, r_ref, torch.bfloat16, None, M)
    print("c client:", stats)


def test_c_stack_client_equals_the_python_stack(tmp_path):
    """tests/c_abi/stack_client.c fills attnres_state from C (flags
    included), runs a 14-layer bf16 stack with and without early loads (the
    same bits, checked there), and checks the fused fold; here the same
    inputs go through the Python binding's StackForward, whose outputs must
    be the client's bit for bit (the two bindings lay the state out alike
    and issue the same launches)."""
    import depth_wise_attention_block_gb300 as A
    from depth_wise_attention_block_gb300.stack import StackForward
    raw = _build_and_run(tmp_path, "stack_client")
    T, d, L, Bs = (int(v) for v in np.frombuffer(raw[:16], dtype=np.int32))
    off = 16

    def take(dtype, n):
        nonlocal off
        a = np.frombuffer(raw, dtype, n, off)
        off += n * np.dtype(dtype).itemsize
        return a

    h0 = torch.from_numpy(take(np.uint16, T * d).astype(np.int16)).view(torch.bfloat16).reshape(T, d).cuda()
    W = torch.from_numpy(take(np.float32, (L + 1) * d).copy()).reshape(L + 1, d).cuda()
    G = torch.from_numpy(take(np.float32, L * d).copy()).reshape(L, d).cuda()
    Sc = torch.from_numpy(take(np.float32, L * d).copy()).reshape(L, d).cuda()
    r_c = take(np.uint16, T * d)
    nw = T * sum(A.attnres_num_sources(l, Bs, L) for l in range(1, L + 2))
    w_c = take(np.float32, nw)
    assert off == len(raw)
    fwd = StackForward(h0, W, G, Sc, L, Bs)
    fwd.run()
    torch.cuda.synchronize()
    r_py = fwd.r.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
    w_py = torch.cat([w.reshape(-1) for w in fwd.weights]).cpu().numpy()
    assert (r_py == r_c).all()
    assert (w_py.view(np.uint32) == w_c.view(np.uint32)).all()
