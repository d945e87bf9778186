"""Tolerances and comparison helpers of the GPU-vs-oracle parity tests.

The bars (all written out here, used by every parity test):

* weights a[t, s] (fp32 on the GPU): |a_gpu - a_ref| <= 1e-5 absolute;
* fp32 outputs r: |r_gpu - r_ref| <= 1e-5 * (|r_ref| + sum_s a_s |h_s|),
  i.e. 1e-5 relative to the condition scale of the weighted sum, so that
  outputs that cancel to near zero do not fail spuriously;
* bf16 outputs r (bf16 storage, fp32 accumulation):
  |r_gpu - r_ref| <= ulp_bf16(r_ref) + 1e-3 * M_t with M_t = max_{s,c}
  |h_s[t, c]| per token (the largest source magnitude of that token).

r_ref and a_ref are the fp64 oracle's results on the very bytes the GPU
read.  Nothing here computes the method itself.

Free-running bf16 stacks (many layers, each side feeding its own stored
outputs forward) cannot meet the 1e-5 weight bar: wherever the GPU's fp32
value and the oracle's fp64 value of a stored tensor straddle a bf16
rounding boundary, the stored values differ by one ulp, and those flips
spread to later layers (measured: ~30% of elements after a few blocks, while
fp32 storage stays within 2e-7).  With one-ulp differences of independent
sign in the sources, the logit difference w.(dh)/rms has standard deviation
at most 2^-7 (ulp <= 2^-7 |h|, w ~ N(0, 1/d) so E[sum_c w_c^2 h_c^2/rms^2] = 1);
the largest of ~10^5 logits is within ~4.7 sigma = 0.037, and a softmax weight
moves by at most about half the largest logit change: 0.018.  So free-running
bf16 stacks use STACK_BF16_A_ATOL = 2e-2 for the weights (a bookkeeping
mistake moves weights by O(0.1-1)); their outputs keep the bf16 bar above.
fp32-storage stacks use the fp32 bars unchanged.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

A_ATOL = 1e-5
R_F32_RTOL = 1e-5
R_BF16_MABS = 1e-3
STACK_BF16_A_ATOL = 2e-2


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 values in the binade of |x| (2^-133 at zero)."""
    _, e = np.frexp(np.abs(x))
    q = np.maximum(e - 8, -133)
    return np.where(x == 0, 2.0 ** -133, np.ldexp(1.0, q))


def oracle_aggregate(H: torch.Tensor, w: torch.Tensor, eps: float, chunk: int = 256):
    """Oracle on a (possibly large) [S, T, d] tensor, token chunk by chunk.
    Returns (r_ref [T, d], a_ref [T, S], cond [T, d], M [T]) in fp64, where
    cond = sum_s a_s |h_s| and M = max_{s,c} |h_s|."""
    S, T, d = H.shape
    w64 = to64(w)
    r = np.empty((T, d))
    a = np.empty((T, S))
    cond = np.empty((T, d))
    M = np.empty(T)
    for t0 in range(0, T, chunk):
        h = to64(H[:, t0:t0 + chunk])
        rr, aa = O.depth_attention(h, w64, eps)
        r[t0:t0 + chunk] = rr
        a[t0:t0 + chunk] = aa
        cond[t0:t0 + chunk] = np.einsum("ts,std->td", aa, np.abs(h))
        M[t0:t0 + chunk] = np.abs(h).max(axis=(0, 2))
    return r, a, cond, M


def oracle_backward(H: torch.Tensor, w: torch.Tensor, dr: torch.Tensor, eps: float, chunk: int = 256):
    """Oracle gradients and their condition scales, token chunk by chunk."""
    S, T, d = H.shape
    dH = np.empty((S, T, d))
    dHs = np.empty((S, T, d))
    dw = np.zeros(d)
    dws = np.zeros(d)
    w64 = to64(w)
    for t0 in range(0, T, chunk):
        h, g = to64(H[:, t0:t0 + chunk]), to64(dr[t0:t0 + chunk])
        a, b = O.depth_attention_backward(h, w64, g, eps)
        sa, sb = O.depth_attention_backward_scales(h, w64, g, eps)
        dH[:, t0:t0 + chunk], dHs[:, t0:t0 + chunk] = a, sa
        dw += b
        dws += sb
    return dH, dw, dHs, dws


def check_weights(a_gpu: np.ndarray, a_ref: np.ndarray) -> float:
    err = np.abs(a_gpu - a_ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= A_ATOL, f"weights off by {worst:.3g} > {A_ATOL}"
    return worst


def check_r(r_gpu: np.ndarray, r_ref: np.ndarray, out_dtype: torch.dtype, cond: np.ndarray | None = None,
            M: np.ndarray | None = None) -> dict:
    """Assert the output bar; return error statistics."""
    err = np.abs(r_gpu - r_ref)
    if out_dtype == torch.float32:
        bound = R_F32_RTOL * (np.abs(r_ref) + cond)
        ratio = err / np.maximum(bound, np.finfo(np.float64).tiny)
        assert (err <= bound).all(), f"fp32 r: worst error {ratio.max():.3g} x the bound"
        return {"max_abs": float(err.max(initial=0)), "worst_ratio": float(ratio.max(initial=0))}
    ulp = ulp_bf16(r_ref)
    bound = ulp + R_BF16_MABS * M[:, None]
    ratio = err / bound
    assert (err <= bound).all(), f"bf16 r: worst error {ratio.max():.3g} x the bound"
    return {"max_abs": float(err.max(initial=0)), "max_ulps": float((err / ulp).max(initial=0)),
            "worst_ratio": float(ratio.max(initial=0))}
