"""Block Attention Residuals (Block AttnRes) depth aggregation for GB300.

A thin Python binding of ``libattnres`` (C ABI in ``include/attnres.h``);
the functions keep the C names.  torch supplies device memory and streams
only: tensors are passed as device pointers, the current torch CUDA stream
is used unless one is given, and every step of the computation runs in the
library's sm_103a kernels.  Importing raises if the library is missing.

What is computed ("Kimi K3 deep-dive series (2): AttnRes and Stable
LatentMoE", §2; Kimi K3 chaptered tutorial, ch. 4.3 Eq. 10):
    a_l = softmax_s(w_l . RMSNorm(h_s)),  r_l = sum_s a_l[s] h_s
over the sources [h_0, b_1 .. b_{n-1}, partial sum of the current block].
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import torch

from . import _native as _N
from ._native import (  # noqa: F401
    ATTNRES_BF16,
    ATTNRES_DEFAULT_EPS,
    ATTNRES_DEVERR_WAIT_TIMEOUT,
    ATTNRES_F32,
    ATTNRES_MAX_BLOCKS,
    ATTNRES_MAX_SOURCES,
    ATTNRES_STATE_EARLY_LOADS,
    AttnresError,
    LIB_PATH,
)

__all__ = [
    "attnres_aggregate", "attnres_aggregate_backward", "attnres_aggregate_backward_workspace_size",
    "attnres_interblock", "attnres_interblock_workspace_size", "attnres_intrablock_step", "attnres_num_sources", "attnres_layer_sources", "attnres_block_step",
    "attnres_layer_step", "attnres_synthetic_layer", "attnres_synthetic_layer_backward", "attnres_fold",
    "attnres_aggregate_fold",
    "attnres_version", "AttnResState",
    "attnres_aggregate_host", "attnres_aggregate_host_workspace_size", "dtype_code", "AttnresError",
]

_DT = {torch.float32: ATTNRES_F32, torch.bfloat16: ATTNRES_BF16}


def dtype_code(dt: torch.dtype) -> int:
    try:
        return _DT[dt]
    except KeyError:
        raise TypeError(f"unsupported dtype {dt}; use float32 or bfloat16") from None


def _dev_ptr(t: torch.Tensor | None, name: str, dtype=None, contiguous=True) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    # the library launches on the current device: another device's memory
    # must never reach its kernels
    cur = torch.cuda.current_device()
    if t.get_device() != cur:
        raise ValueError(f"{name} is on {t.device} but the current device is cuda:{cur}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream) -> int:
    if stream is None:
        # the current stream's handle without building a Stream object
        if _RAW_STREAM is not None:
            return _RAW_STREAM(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def attnres_version() -> int:
    return _N.lib.attnres_version()


def attnres_num_sources(layer_idx: int, block_size: int, num_layers: int) -> int:
    """Sources of layer `layer_idx` (L+1 = the final output aggregation)."""
    return _N.check(_N.lib.attnres_num_sources(layer_idx, block_size, num_layers), "attnres_num_sources")


def attnres_aggregate(sources: Sequence[torch.Tensor] | torch.Tensor, w_l: torch.Tensor, out_r: torch.Tensor,
                      out_weights: torch.Tensor | None = None, eps: float = ATTNRES_DEFAULT_EPS,
                      dev_err: torch.Tensor | None = None, stream=None) -> None:
    """One layer of depth-wise attention.

    sources: S CUDA tensors [T, d] (float32 or bfloat16, one dtype), or one
    [S, T, d] tensor; w_l: [d] float32; out_r: [T, d] float32/bfloat16;
    out_weights: [T, S] float32 or None; dev_err: int32 [1] or None.
    """
    if isinstance(sources, torch.Tensor) and sources.dim() == 3 and not sources.is_contiguous():
        sources = list(sources.unbind(0))  # e.g. every other source: each slice checked below
    if isinstance(sources, torch.Tensor):
        # one contiguous [S, T, d] tensor: checked once, source s at base + s * T * d
        if sources.dim() != 3:
            raise ValueError("a stacked sources tensor must be [S, T, d]")
        S, T, d = sources.shape
        dt = sources.dtype
        base = _dev_ptr(sources, "sources")
        step = T * d * sources.element_size()
        ptrs = (ctypes.c_void_p * S)(*[base + i * step for i in range(S)]) if S else None
    else:
        srcs = list(sources)
        S = len(srcs)
        if not srcs:
            raise ValueError("need at least one source")
        T, d = srcs[0].shape
        dt = srcs[0].dtype
        for i, s in enumerate(srcs):
            if s.shape != (T, d) or s.dtype != dt:
                raise ValueError(f"source {i}: expected [{T}, {d}] {dt}, got {list(s.shape)} {s.dtype}")
        ptrs = (ctypes.c_void_p * S)(*[_dev_ptr(s, f"sources[{i}]") for i, s in enumerate(srcs)])
    if S < 1:
        raise ValueError("need at least one source")
    if out_r.shape != (T, d):
        raise ValueError("out_r must be [T, d]")
    if out_weights is not None and out_weights.shape != (T, S):
        raise ValueError("out_weights must be [T, S]")
    rc = _N.lib.attnres_aggregate(
        ptrs, S, T, d, dtype_code(dt), _dev_ptr(w_l, "w_l", torch.float32), float(eps),
        _dev_ptr(out_r, "out_r"), dtype_code(out_r.dtype), _dev_ptr(out_weights, "out_weights", torch.float32),
        _dev_ptr(dev_err, "dev_err", torch.int32), _stream_ptr(stream))
    _N.check(rc, "attnres_aggregate")


def attnres_aggregate_backward_workspace_size(T: int, d: int) -> int:
    """Bytes of device workspace attnres_aggregate_backward needs."""
    return _N.check(_N.lib.attnres_aggregate_backward_workspace_size(T, d), "attnres_aggregate_backward_workspace_size")


def attnres_aggregate_backward(sources: Sequence[torch.Tensor] | torch.Tensor, w_l: torch.Tensor,
                               grad_r: torch.Tensor, grad_sources: Sequence[torch.Tensor] | torch.Tensor,
                               grad_w: torch.Tensor, workspace: torch.Tensor | None = None,
                               eps: float = ATTNRES_DEFAULT_EPS, accumulate: bool = False,
                               dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Gradients of attnres_aggregate with respect to its sources and w_l
    (the forward is recomputed).  grad_sources: S tensors [T, d] (or one
    [S, T, d]) of the sources' dtype, overwritten or (accumulate) added to;
    grad_w: [d] float32, overwritten.  workspace: a device buffer of at least
    attnres_aggregate_backward_workspace_size(T, d) bytes (allocated here
    through torch when None)."""
    srcs = list(sources.unbind(0)) if isinstance(sources, torch.Tensor) else list(sources)
    grads = list(grad_sources.unbind(0)) if isinstance(grad_sources, torch.Tensor) else list(grad_sources)
    if len(grads) != len(srcs):
        raise ValueError("need one gradient buffer per source")
    T, d = srcs[0].shape
    dt = srcs[0].dtype
    for i, t in enumerate(srcs + grads + [grad_r]):
        if t.shape != (T, d) or t.dtype != dt:
            raise ValueError(f"tensor {i}: expected [{T}, {d}] {dt}")
    if workspace is None:
        nbytes = attnres_aggregate_backward_workspace_size(T, d)
        workspace = torch.empty(max(1, nbytes // 4), dtype=torch.float32, device=srcs[0].device)
    S = len(srcs)
    sp = (ctypes.c_void_p * S)(*[_dev_ptr(t, f"sources[{i}]") for i, t in enumerate(srcs)])
    gp = (ctypes.c_void_p * S)(*[_dev_ptr(t, f"grad_sources[{i}]") for i, t in enumerate(grads)])
    rc = _N.lib.attnres_aggregate_backward(
        sp, S, T, d, dtype_code(dt), _dev_ptr(w_l, "w_l", torch.float32), float(eps), _dev_ptr(grad_r, "grad_r"),
        gp, int(bool(accumulate)), _dev_ptr(grad_w, "grad_w", torch.float32), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dev_ptr(dev_err, "dev_err", torch.int32), _stream_ptr(stream))
    _N.check(rc, "attnres_aggregate_backward")


def attnres_interblock_workspace_size(n: int, T: int, d: int, dtype: torch.dtype, Q: int) -> int:
    """Bytes of workspace attnres_interblock's tensor-core logits need (0: the
    path does not apply, e.g. fp32 sources)."""
    return _N.check(_N.lib.attnres_interblock_workspace_size(int(n), int(T), int(d), dtype_code(dtype), int(Q)),
                    "attnres_interblock_workspace_size")


def attnres_interblock(sources: Sequence[torch.Tensor], w_queries: Sequence[torch.Tensor] | torch.Tensor,
                       out_r: torch.Tensor, out_lse: torch.Tensor, out_weights: torch.Tensor | None = None,
                       eps: float = ATTNRES_DEFAULT_EPS, workspace: torch.Tensor | None = None,
                       tensor_cores: bool = True, dev_err: torch.Tensor | None = None, stream=None,
                       out_r0: torch.Tensor | None = None, out_weights0: torch.Tensor | None = None) -> None:
    """Phase 1 of the two-phase schedule: the n cached sources aggregated for
    Q queries at once.  out_r [Q, T, d] fp32, out_lse [Q, T] fp32,
    out_weights [Q, T, n] fp32 or None.  With tensor_cores (bf16 sources, d
    a multiple of 64) the logits run on the tensor cores in a workspace of
    attnres_interblock_workspace_size bytes (allocated here through torch
    when None); tensor_cores=False keeps every step on the CUDA cores.
    out_r0 [T, d] of the sources' dtype and out_weights0 [T, n] fp32 (or
    None): the block's first layer's output and weights, written here."""
    srcs = list(sources)
    qs = list(w_queries.unbind(0)) if isinstance(w_queries, torch.Tensor) else list(w_queries)
    T, d = srcs[0].shape
    dt = srcs[0].dtype
    ws_ptr, ws_bytes = None, 0
    if tensor_cores:
        need = attnres_interblock_workspace_size(len(srcs), T, d, dt, len(qs))
        if need > 0:
            if workspace is None:
                workspace = torch.empty(need, dtype=torch.uint8, device=srcs[0].device)
            ws_ptr = _dev_ptr(workspace, "workspace")
            ws_bytes = workspace.numel() * workspace.element_size()
    sp = (ctypes.c_void_p * len(srcs))(*[_dev_ptr(t, f"sources[{i}]") for i, t in enumerate(srcs)])
    qp = (ctypes.c_void_p * len(qs))(*[_dev_ptr(q, f"w_queries[{i}]", torch.float32) for i, q in enumerate(qs)])
    rc = _N.lib.attnres_interblock(sp, len(srcs), T, d, dtype_code(dt), qp, len(qs), float(eps),
                                   _dev_ptr(out_r, "out_r", torch.float32), _dev_ptr(out_lse, "out_lse", torch.float32),
                                   _dev_ptr(out_weights, "out_weights", torch.float32),
                                   _dev_ptr(out_r0, "out_r0", dt), _dev_ptr(out_weights0, "out_weights0", torch.float32),
                                   ws_ptr, ws_bytes, _dev_ptr(dev_err, "dev_err", torch.int32), _stream_ptr(stream))
    _N.check(rc, "attnres_interblock")


def attnres_intrablock_step(state: "AttnResState", F_prev: torch.Tensor | None, w_l: torch.Tensor, layer_idx: int,
                            r_inter: torch.Tensor, lse_inter: torch.Tensor, a_inter: torch.Tensor | None,
                            out_r: torch.Tensor, out_weights: torch.Tensor | None = None,
                            dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Phase 2 of the two-phase schedule for one layer (see include/attnres.h)."""
    rc = _N.lib.attnres_intrablock_step(
        ctypes.byref(state.struct), _dev_ptr(F_prev, "F_prev", state.h0.dtype), _dev_ptr(w_l, "w_l", torch.float32),
        layer_idx, _dev_ptr(r_inter, "r_inter", torch.float32), _dev_ptr(lse_inter, "lse_inter", torch.float32),
        _dev_ptr(a_inter, "a_inter", torch.float32), _dev_ptr(out_r, "out_r", state.h0.dtype),
        _dev_ptr(out_weights, "out_weights", torch.float32), _dev_ptr(dev_err, "dev_err", torch.int32),
        _stream_ptr(stream))
    _N.check(rc, "attnres_intrablock_step")


class AttnResState:
    """Resident depth sources of one batch (embedding, block sums, partial).

    Holds the torch buffers (so they outlive the C struct's pointers) and the
    `attnres_state` struct the C ABI updates.
    """

    def __init__(self, h0: torch.Tensor, block_reps: Sequence[torch.Tensor], partial: torch.Tensor,
                 num_layers: int, block_size: int, eps: float = ATTNRES_DEFAULT_EPS, early_loads: bool = False):
        T, d = h0.shape
        for i, b in enumerate(list(block_reps) + [partial]):
            if b.shape != (T, d) or b.dtype != h0.dtype:
                raise ValueError(f"state buffer {i} must be [{T}, {d}] {h0.dtype}")
        self.h0, self.block_reps, self.partial = h0, list(block_reps), partial
        self.num_layers, self.block_size = num_layers, block_size
        self.struct = _N.AttnresState()
        reps = (ctypes.c_void_p * max(1, len(self.block_reps)))(
            *[_dev_ptr(b, f"block_reps[{i}]") for i, b in enumerate(self.block_reps)])
        rc = _N.lib.attnres_state_init(ctypes.byref(self.struct), _dev_ptr(h0, "h0"), reps, len(self.block_reps),
                                       _dev_ptr(partial, "partial"), T, d, dtype_code(h0.dtype), num_layers,
                                       block_size, float(eps))
        _N.check(rc, "attnres_state_init")
        # ATTNRES_STATE_EARLY_LOADS: see include/attnres.h for when it is safe
        self.struct.flags = ATTNRES_STATE_EARLY_LOADS if early_loads else 0

    @classmethod
    def allocate(cls, h0: torch.Tensor, num_layers: int, block_size: int, eps: float = ATTNRES_DEFAULT_EPS,
                 early_loads: bool = False):
        n_blocks = -(-num_layers // block_size)
        reps = [torch.empty_like(h0) for _ in range(n_blocks)]
        return cls(h0, reps, torch.empty_like(h0), num_layers, block_size, eps, early_loads)

    @property
    def folded(self) -> int:
        return self.struct.folded

    def reset(self) -> None:
        _N.check(_N.lib.attnres_state_reset(ctypes.byref(self.struct)), "attnres_state_reset")

    def resume(self, folded: int) -> None:
        """Take up the stack after layer `folded` (v_1 .. v_folded already in
        the buffers, e.g. received at a pipeline stage boundary); see
        attnres_state_resume."""
        _N.check(_N.lib.attnres_state_resume(ctypes.byref(self.struct), int(folded)), "attnres_state_resume")


def attnres_layer_sources(state: AttnResState, layer_idx: int) -> list[int]:
    """Device pointers of layer `layer_idx`'s sources, in order."""
    out = (ctypes.c_void_p * ATTNRES_MAX_SOURCES)()
    n = ctypes.c_int(0)
    _N.check(_N.lib.attnres_layer_sources(ctypes.byref(state.struct), layer_idx, out, ctypes.byref(n)),
             "attnres_layer_sources")
    return [out[i] for i in range(n.value)]


def attnres_block_step(state: AttnResState, F_out: torch.Tensor, layer_idx: int,
                       dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Fold layer `layer_idx`'s output into the partial sum / block representation."""
    rc = _N.lib.attnres_block_step(ctypes.byref(state.struct), _dev_ptr(F_out, "F_out", state.h0.dtype), layer_idx,
                                   _dev_ptr(dev_err, "dev_err", torch.int32), _stream_ptr(stream))
    _N.check(rc, "attnres_block_step")


def attnres_layer_step(state: AttnResState, F_prev: torch.Tensor | None, w_l: torch.Tensor, layer_idx: int,
                       out_r: torch.Tensor, out_weights: torch.Tensor | None = None,
                       dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Fused: fold F_prev = v_{l-1}, then aggregate layer `layer_idx`.
    F_prev None: nothing left to fold (layer 1, or a resumed state)."""
    rc = _N.lib.attnres_layer_step(
        ctypes.byref(state.struct), _dev_ptr(F_prev, "F_prev", state.h0.dtype),
        _dev_ptr(w_l, "w_l", torch.float32), layer_idx, _dev_ptr(out_r, "out_r", state.h0.dtype),
        _dev_ptr(out_weights, "out_weights", torch.float32), _dev_ptr(dev_err, "dev_err", torch.int32),
        _stream_ptr(stream))
    _N.check(rc, "attnres_layer_step")


def attnres_synthetic_layer(x: torch.Tensor, g: torch.Tensor, s: torch.Tensor, out: torch.Tensor,
                            stream=None) -> None:
    """Stand-in layer body out = tanh(x * g) * s (drives a stack; not the method)."""
    T, d = x.shape
    rc = _N.lib.attnres_synthetic_layer(_dev_ptr(x, "x"), _dev_ptr(g, "g", torch.float32),
                                        _dev_ptr(s, "s", torch.float32), _dev_ptr(out, "out", x.dtype), T, d,
                                        dtype_code(x.dtype), _stream_ptr(stream))
    _N.check(rc, "attnres_synthetic_layer")


def attnres_synthetic_layer_backward(x: torch.Tensor, g: torch.Tensor, s: torch.Tensor, grad_out_a: torch.Tensor,
                                     grad_out_b: torch.Tensor | None, grad_x: torch.Tensor, stream=None) -> None:
    """Gradient of the stand-in body: grad_x = (grad_out_a + grad_out_b) * (1 - tanh(x g)^2) * g * s."""
    T, d = x.shape
    for name, t in (("grad_out_a", grad_out_a), ("grad_out_b", grad_out_b), ("grad_x", grad_x)):
        if t is not None and t.shape != (T, d):
            raise ValueError(f"{name} must be [T, d]")
    rc = _N.lib.attnres_synthetic_layer_backward(
        _dev_ptr(x, "x"), _dev_ptr(g, "g", torch.float32), _dev_ptr(s, "s", torch.float32),
        _dev_ptr(grad_out_a, "grad_out_a", x.dtype), _dev_ptr(grad_out_b, "grad_out_b", x.dtype),
        _dev_ptr(grad_x, "grad_x", x.dtype), T, d, dtype_code(x.dtype), _stream_ptr(stream))
    _N.check(rc, "attnres_synthetic_layer_backward")


def attnres_fold(prev: torch.Tensor | None, F: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    """Block bookkeeping on plain buffers: dst = prev + F (one rounding), or F when prev is None."""
    T, d = F.shape
    if dst.shape != (T, d) or (prev is not None and prev.shape != (T, d)):
        raise ValueError("prev, F and dst must all be [T, d]")
    rc = _N.lib.attnres_fold(_dev_ptr(prev, "prev", F.dtype), _dev_ptr(F, "F"), _dev_ptr(dst, "dst", F.dtype), T, d,
                             dtype_code(F.dtype), _stream_ptr(stream))
    _N.check(rc, "attnres_fold")


def attnres_aggregate_fold(sources: Sequence[torch.Tensor], prev: torch.Tensor | None, F: torch.Tensor,
                           dst: torch.Tensor, w_l: torch.Tensor, out_r: torch.Tensor,
                           out_weights: torch.Tensor | None = None, eps: float = ATTNRES_DEFAULT_EPS,
                           early_loads: bool = False, dev_err: torch.Tensor | None = None, stream=None) -> None:
    """One layer over the stored sources and the partial sum dst = prev + F
    (or F) formed and stored in the same launch; see include/attnres.h.
    Every row [T, d] of F's dtype; out_r the same; out_weights
    [T, len(sources) + 1] float32 or None.  early_loads: see
    ATTNRES_STATE_EARLY_LOADS (only when the kernel just before writes
    nothing this call reads but F)."""
    T, d = F.shape
    srcs = list(sources)
    for i, t in enumerate(srcs + [dst] + ([prev] if prev is not None else []) + [out_r]):
        if t.shape != (T, d) or t.dtype != F.dtype:
            raise ValueError(f"row {i}: expected [{T}, {d}] {F.dtype}, got {list(t.shape)} {t.dtype}")
    if out_weights is not None and out_weights.shape != (T, len(srcs) + 1):
        raise ValueError("out_weights must be [T, n_stored + 1]")
    ptrs = (ctypes.c_void_p * max(1, len(srcs)))(*[_dev_ptr(t, f"sources[{i}]") for i, t in enumerate(srcs)])
    rc = _N.lib.attnres_aggregate_fold(
        ptrs, len(srcs), _dev_ptr(prev, "prev"), _dev_ptr(F, "F"), _dev_ptr(dst, "dst"), T, d, dtype_code(F.dtype),
        _dev_ptr(w_l, "w_l", torch.float32), float(eps), _dev_ptr(out_r, "out_r"),
        _dev_ptr(out_weights, "out_weights", torch.float32), ATTNRES_STATE_EARLY_LOADS if early_loads else 0,
        _dev_ptr(dev_err, "dev_err", torch.int32), _stream_ptr(stream))
    _N.check(rc, "attnres_aggregate_fold")


def attnres_debug_wait_test(wait_limit_ns: int, withhold_row: int) -> None:
    """Diagnostic: make the ring kernels' bounded waits run out (withhold_row
    0..7 of every CTA's first token is armed without a copy; waits limited to
    wait_limit_ns).  (0, -1) restores normal operation."""
    _N.check(_N.lib.attnres_debug_wait_test(int(wait_limit_ns), int(withhold_row)), "attnres_debug_wait_test")


def _host_ptr(t: torch.Tensor | None, name: str, dtype=None) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def attnres_aggregate_host_workspace_size(S: int, chunk_tokens: int, d: int, src_dtype: torch.dtype,
                                          out_dtype: torch.dtype, with_weights: bool = True, slots: int = 2) -> int:
    """Bytes of device workspace attnres_aggregate_host needs for `slots`
    staging slots of chunk_tokens tokens."""
    return _N.check(_N.lib.attnres_aggregate_host_workspace_size(
        int(S), int(chunk_tokens), int(d), dtype_code(src_dtype), dtype_code(out_dtype), int(bool(with_weights)),
        int(slots)), "attnres_aggregate_host_workspace_size")


def attnres_aggregate_host(sources_host: Sequence[torch.Tensor] | torch.Tensor, w_host: torch.Tensor,
                           r_host: torch.Tensor, weights_host: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, chunk_tokens: int = 1024,
                           eps: float = ATTNRES_DEFAULT_EPS, dev_err: torch.Tensor | None = None,
                           stream=None) -> None:
    """attnres_aggregate with sources, query and outputs in host memory.

    sources_host: S CPU tensors [T, d] (float32 or bfloat16, one dtype,
    pinned for full speed) or one [S, T, d] CPU tensor; w_host: [d] float32;
    r_host: [T, d] float32/bfloat16; weights_host: [T, S] float32 or None;
    workspace: a CUDA tensor of at least attnres_aggregate_host_workspace_size
    bytes (None: two slots are allocated through torch).  The library streams
    token chunks through the workspace's staging slots; synchronise `stream`
    (default: the current stream) before reading r_host.
    """
    if isinstance(sources_host, torch.Tensor):
        if sources_host.dim() != 3:
            raise ValueError("a stacked sources tensor must be [S, T, d]")
        srcs = list(sources_host.unbind(0))
    else:
        srcs = list(sources_host)
    if not srcs:
        raise ValueError("need at least one source")
    T, d = srcs[0].shape
    dt = srcs[0].dtype
    for i, s in enumerate(srcs):
        if s.shape != (T, d) or s.dtype != dt:
            raise ValueError(f"source {i}: expected [{T}, {d}] {dt}, got {list(s.shape)} {s.dtype}")
    ptrs = (ctypes.c_void_p * len(srcs))(*[_host_ptr(s, f"sources_host[{i}]") for i, s in enumerate(srcs)])
    if r_host.shape != (T, d):
        raise ValueError("r_host must be [T, d]")
    if weights_host is not None and weights_host.shape != (T, len(srcs)):
        raise ValueError("weights_host must be [T, S]")
    if w_host.shape != (d,):
        raise ValueError("w_host must be [d]")
    if workspace is None:
        nbytes = attnres_aggregate_host_workspace_size(len(srcs), max(1, min(int(chunk_tokens), T)), d, dt,
                                                       r_host.dtype, weights_host is not None, 2)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=torch.cuda.current_device())
    rc = _N.lib.attnres_aggregate_host(
        ptrs, len(srcs), T, d, dtype_code(dt), _host_ptr(w_host, "w_host", torch.float32), float(eps),
        _host_ptr(r_host, "r_host"), dtype_code(r_host.dtype), _host_ptr(weights_host, "weights_host", torch.float32),
        int(chunk_tokens), _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev_ptr(dev_err, "dev_err", torch.int32), _stream_ptr(stream))
    _N.check(rc, "attnres_aggregate_host")
