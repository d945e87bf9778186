"""Seeded synthetic inputs for Block AttnRes depth aggregation.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic (no RMSNorm, no softmax, no sums over sources).  Both the
fp64 oracle (through the tests and the bench) and the CUDA path are fed the
exact bytes produced here, so the two sides never share computation.

Shapes and distributions follow the workloads the pages describe for the
93-layer Kimi K3 model (hidden size d = 7168, 12-layer blocks, at most nine
sources per token): "LLM Atlas · Kimi K3", §03 Table 1 and §07 Attention
Residuals; "Kimi K3 deep-dive (2): AttnRes and Stable LatentMoE", §3.

Draw order inside one generator (a ``torch.Generator`` seeded with the
workload seed, on the device the tensors are made on):

1. single-layer workloads: (outlier selection, long-context workload only),
   then the sources in index order, then the pseudo-query ``w``;
2. stack workloads: ``h_0``, then ``w_1 .. w_{L+1}``, then ``g_1 .. g_L``,
   then ``s_1 .. s_L``.

A CPU generator and a CUDA generator give different numbers for one seed;
each test feeds both sides the tensors of one generator, so that does not
matter for parity.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

D_MODEL = 7168          # K3 hidden size
NUM_LAYERS = 93         # K3 transformer layers
BLOCK_SIZE = 12         # layers per AttnRes block (12 x 7 + 9)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


@dataclass
class SingleLayer:
    """One aggregation problem: sources H [S, T, d] and pseudo-query w [d]."""
    H: torch.Tensor                 # [S, T, d], float32 or bfloat16
    w: torch.Tensor                 # [d], float32
    outlier_tokens: torch.Tensor | None = None   # [n] int64 (long-context only)
    outlier_sources: torch.Tensor | None = None  # [n] int64


def full_fp32(T: int = 64, d: int = 256, sigmas=(0.5, 1.0, 2.0, 4.0), seed: int = 0,
              device="cpu") -> SingleLayer:
    """Full AttnRes, one layer, fp32: h_s ~ N(0, sigma_s^2), w ~ N(0, 1/d)."""
    g = _gen(seed, device)
    H = torch.empty((len(sigmas), T, d), dtype=torch.float32, device=device)
    for s, sig in enumerate(sigmas):
        H[s] = torch.randn((T, d), generator=g, device=device) * float(sig)
    w = torch.randn((d,), generator=g, device=device) / math.sqrt(d)
    return SingleLayer(H=H, w=w)


def block_sigmas(num_blocks: int = 7) -> list[float]:
    """Per-source std of the nine-source workload: h_0 ~ N(0,1), block sum k
    ~ N(0, (0.5 sqrt k)^2) for k = 1..num_blocks, partial sum ~ N(0, 4)."""
    return [1.0] + [0.5 * math.sqrt(k) for k in range(1, num_blocks + 1)] + [2.0]


def block_bf16(T: int = 4096, d: int = D_MODEL, seed: int = 1, device="cpu",
               outlier_frac: float = 0.0, outlier_scale: float = 50.0,
               num_blocks: int = 7, src_dtype=torch.bfloat16) -> SingleLayer:
    """Block AttnRes single layer: S = num_blocks + 2 sources stored as one
    [S, T, d] slab in the order [h_0, b_1 .. b_num_blocks, partial].

    With ``outlier_frac > 0`` a fraction of the tokens (drawn without
    replacement) get one source (drawn uniformly) multiplied by
    ``outlier_scale`` before the cast to ``src_dtype``.
    """
    g = _gen(seed, device)
    sig = block_sigmas(num_blocks)
    S = len(sig)
    otok = osrc = None
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * T))
        otok = torch.randperm(T, generator=g, device=device)[:n_out]
        osrc = torch.randint(0, S, (n_out,), generator=g, device=device)
    H = torch.empty((S, T, d), dtype=src_dtype, device=device)
    for s in range(S):
        x = torch.randn((T, d), generator=g, device=device, dtype=torch.float32)
        x.mul_(sig[s])
        if otok is not None:
            rows = otok[osrc == s]
            if rows.numel():
                x[rows] *= outlier_scale
        H[s] = x.to(src_dtype)
        del x
    w = torch.randn((d,), generator=g, device=device) / math.sqrt(d)
    return SingleLayer(H=H, w=w, outlier_tokens=otok, outlier_sources=osrc)


def full_bf16(T: int = 2048, d: int = D_MODEL, S: int = 94, seed: int = 5, device="cpu",
              out_sigma: float = 0.1) -> SingleLayer:
    """Full AttnRes single layer over S sources stored as one bf16 [S, T, d]
    slab: the embedding h_0 ~ N(0, 1) and S - 1 earlier layer outputs
    ~ N(0, out_sigma^2) (the stand-in body's outputs are bounded by its
    scale s <= 0.2); w ~ N(0, 1/d)."""
    g = _gen(seed, device)
    H = torch.empty((S, T, d), dtype=torch.bfloat16, device=device)
    for s in range(S):
        x = torch.randn((T, d), generator=g, device=device, dtype=torch.float32)
        if s > 0:
            x.mul_(out_sigma)
        H[s] = x.to(torch.bfloat16)
        del x
    w = torch.randn((d,), generator=g, device=device) / math.sqrt(d)
    return SingleLayer(H=H, w=w)


@dataclass
class Stack:
    """Inputs of a synthetic L-layer Block AttnRes stack forward."""
    h0: torch.Tensor      # [T, d] embedding, storage dtype
    W: torch.Tensor       # [L + 1, d] float32 pseudo-queries; row L is the final aggregation's
    G: torch.Tensor       # [L, d] float32 gains of the synthetic layer function
    Sc: torch.Tensor      # [L, d] float32 scales of the synthetic layer function
    num_layers: int
    block_size: int


def stack(T: int = 2048, d: int = D_MODEL, num_layers: int = NUM_LAYERS,
          block_size: int = BLOCK_SIZE, seed: int = 2, device="cpu",
          dtype=torch.bfloat16) -> Stack:
    """h_0 ~ N(0,1); w_l ~ N(0, 1/d) for l = 1..L+1; g_l ~ N(0,1);
    s_l ~ U(0.05, 0.2), all per channel."""
    g = _gen(seed, device)
    h0 = torch.randn((T, d), generator=g, device=device).to(dtype)
    W = torch.randn((num_layers + 1, d), generator=g, device=device) / math.sqrt(d)
    G = torch.randn((num_layers, d), generator=g, device=device)
    Sc = 0.05 + 0.15 * torch.rand((num_layers, d), generator=g, device=device)
    return Stack(h0=h0, W=W, G=G, Sc=Sc, num_layers=num_layers, block_size=block_size)


# The five named workloads (sizes, seeds) ------------------------------------

def full_T64_d256():
    """Full AttnRes, one layer, fp32, T=64, d=256, S=4 (seed 0)."""
    return full_fp32(T=64, d=256, seed=0, device="cpu")


def block_T4096_d7168(device="cuda"):
    """Block AttnRes, one layer, bf16, T=4096, d=7168, S=9 (seed 1)."""
    return block_bf16(T=4096, d=D_MODEL, seed=1, device=device)


def stack_T2048(device="cuda"):
    """93-layer prefill stack, bf16, T=2048, d=7168, block size 12 (seed 2)."""
    return stack(T=2048, seed=2, device=device)


def stack_T64(device="cuda"):
    """93-layer decode-shaped stack, bf16, T=64, d=7168, block size 12 (seed 3)."""
    return stack(T=64, seed=3, device=device)


def block_T131072_d7168(device="cuda"):
    """Long-context single layer, bf16, T=131072, d=7168, S=9, x50 outliers on 1% (seed 4)."""
    return block_bf16(T=131072, d=D_MODEL, seed=4, device=device, outlier_frac=0.01)
