"""fp64 reference definitions of (Block) Attention Residuals.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path, and sharing no code with the CUDA kernels.

Sources cited (page title, then the section / equation on it):

* [Deep-dive 2] "Kimi K3 deep-dive series (2): AttnRes and Stable LatentMoE",
  §1 (plain residual), §2 (pseudo-code and the a_l / r_l formula), §2.1 (the
  four-source worked example), §3 (Block AttnRes, nine sources).
* [Tutorial] Kimi K3 chaptered tutorial (kimi.papertok.ai), ch. 0.11
  (RMSNorm: square, mean, square root), ch. 4.2 (Eq. 8-9: pseudo-query,
  keys = values = layer outputs, phi(q, k) = exp(q^T RMSNorm(k))), ch. 4.3
  (Eq. 10: the two-case value list, the final output aggregating all block
  representations), ch. 4.5 (12-layer blocks, incomplete last block, nine
  sources counting the embedding).
* [Parts 6] "Kimi K3 model structure (6): inputs and parts", list of odd
  facts (RMSNorm eps = 1e-5 model-wide).
* [Atlas] "LLM Atlas · Kimi K3", §07 Attention Residuals (alpha_{i->l} and
  h_l = sum_i alpha v_i), §28 workbench "save per block, not per layer"
  (ceil(L/S) + embedding sources), and the reduced study's train-time forward
  intervention (uniform mixer: zero logits give the mean of the sources).

Everything is float64.  Inputs of any float dtype are widened exactly
(bf16 and fp32 values are exactly representable in fp64).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Sequence

import numpy as np

EPS = 1e-5  # [Parts 6]: RMSNorm eps is 1e-5 throughout the model


# --------------------------------------------------------------------------
# One aggregation: a_l = softmax(w_l RMSNorm(H)^T), r_l = a_l H   [Deep-dive 2 §2]
# --------------------------------------------------------------------------

def rms(h: np.ndarray, eps: float = EPS) -> np.ndarray:
    """Root mean square over the last axis, eps added to the mean square.

    [Tutorial ch. 0.11]: square each value, take the mean, take the square
    root.  The eps of [Parts 6] goes inside the root (the usual RMSNorm
    placement; the pages do not print the formula)."""
    h = np.asarray(h, dtype=np.float64)
    return np.sqrt(np.mean(h * h, axis=-1) + eps)


def rmsnorm(h: np.ndarray, eps: float = EPS) -> np.ndarray:
    """RMSNorm with no learned gain, as in the pseudo-code of [Deep-dive 2 §2]."""
    h = np.asarray(h, dtype=np.float64)
    return h / rms(h, eps)[..., None]


def depth_attention(H: Sequence[np.ndarray] | np.ndarray, w: np.ndarray,
                    eps: float = EPS) -> tuple[np.ndarray, np.ndarray]:
    """Depth-wise attention of one layer over its sources.

    H: the S sources, stacked as [S, T, d] (or a list of S arrays [T, d]);
    w: the layer's pseudo-query [d].
    Returns (r [T, d], a [T, S]), both float64:

        keys   = RMSNorm(H)                       (per source row, no gain)
        logits = w . keys                          (no temperature)
        a      = softmax over the S sources
        r      = sum_s a_s H_s                     (values are the raw sources)

    [Deep-dive 2 §2] pseudo-code and formula; [Tutorial ch. 4.2] Eq. 8-9;
    [Atlas §07] alpha_{i->l}.  The softmax subtracts the per-token maximum
    logit first, which leaves it unchanged mathematically.
    """
    H = np.stack([np.asarray(h, dtype=np.float64) for h in H]) if not isinstance(H, np.ndarray) \
        else np.asarray(H, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    if H.ndim != 3:
        raise ValueError("H must be [S, T, d]")
    keys = rmsnorm(H, eps)                                   # [S, T, d]
    logits = np.einsum("std,d->ts", keys, w)                 # [T, S]
    logits = logits - logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    a = e / e.sum(axis=1, keepdims=True)                     # [T, S]
    r = np.einsum("ts,std->td", a, H)                        # [T, d]
    return r, a


def depth_attention_lse(H: np.ndarray, w: np.ndarray, eps: float = EPS):
    """depth_attention plus the log-sum-exp of the logits (lse [T]): the
    summary of a set of sources that a later online-softmax merge needs."""
    H = np.asarray(H, dtype=np.float64)
    r, a = depth_attention(H, w, eps)
    z = np.einsum("std,d->ts", rmsnorm(H, eps), np.asarray(w, np.float64))
    m = z.max(axis=1)
    return r, a, m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def merge_partial_softmax(r1, lse1, r2, lse2):
    """Online-softmax merge of two disjoint source sets ([Tutorial] ch. 4.4):
    given each set's normalised weighted sum r_i and log-sum-exp lse_i, the
    aggregation over the union is  (e^{lse1} r1 + e^{lse2} r2) /
    (e^{lse1} + e^{lse2}),  evaluated with the larger lse subtracted."""
    lse1, lse2 = np.asarray(lse1, np.float64), np.asarray(lse2, np.float64)
    m = np.maximum(lse1, lse2)
    c1, c2 = np.exp(lse1 - m), np.exp(lse2 - m)
    den = c1 + c2
    r = (c1[:, None] * np.asarray(r1, np.float64) + c2[:, None] * np.asarray(r2, np.float64)) / den[:, None]
    return r, c1 / den, c2 / den


def _backward_core(H: np.ndarray, w: np.ndarray, dr: np.ndarray, eps: float, bump: dict | None = None) -> dict:
    """The backward of one layer, per token, step by step (float64).

    With rho_s = rms(h_s), z_s = (w . h_s) / rho_s, a = softmax(z),
    r = sum_s a_s h_s, the chain rule gives, per token:
        g_s   = dr . h_s,             gbar = sum_s a_s g_s
        dz_s  = a_s (g_s - gbar)                       (softmax)
        alpha_s = dz_s / rho_s,       beta_s = alpha_s z_s / (d rho_s)
        dh_s  = a_s dr + alpha_s w - beta_s h_s        (values; logit, with
                                                        d rho_s / d h_s = h_s / (d rho_s))
        dw   += sum_s alpha_s h_s
    `bump` adds a given [S, T] (or [1, T] for gbar) array to one of the
    intermediate quantities ss (= sum_c h_sc^2), g, z, a, gbar, dz, alpha,
    beta as it is formed, so that the sensitivity of the gradients to each can be
    taken by differences.  Returns the intermediates, dH [S, T, d] and the
    per-token contributions to dw, dw_tok [T, d]."""
    b = bump or {}
    S, T, d = H.shape
    ss = np.einsum("std,std->st", H, H) + b.get("ss", 0.0)
    p = np.einsum("std,d->st", H, w)
    g = np.einsum("std,td->st", H, dr) + b.get("g", 0.0)
    rho = np.sqrt(ss / d + eps)
    z = p / rho + b.get("z", 0.0)
    m = z.max(axis=0, keepdims=True)
    e = np.exp(z - m)
    a = e / e.sum(axis=0, keepdims=True) + b.get("a", 0.0)   # [S, T]
    gbar = (a * g).sum(axis=0, keepdims=True) + b.get("gbar", 0.0)
    dz = a * (g - gbar) + b.get("dz", 0.0)
    alpha = dz / rho + b.get("alpha", 0.0)
    beta = alpha * z / (d * rho) + b.get("beta", 0.0)
    dH = a[:, :, None] * dr[None] + alpha[:, :, None] * w[None, None, :] - beta[:, :, None] * H
    dw_tok = np.einsum("st,std->td", alpha, H)
    return dict(ss=ss, p=p, g=g, rho=rho, z=z, m=m, a=a, gbar=gbar, dz=dz, alpha=alpha, beta=beta,
                dH=dH, dw_tok=dw_tok)


def depth_attention_backward(H: np.ndarray, w: np.ndarray, dr: np.ndarray,
                             eps: float = EPS) -> tuple[np.ndarray, np.ndarray]:
    """Gradients of one depth-wise attention layer, recomputing its forward.

    H [S, T, d] sources, w [d] pseudo-query, dr [T, d] gradient of the loss
    with respect to r.  Returns (dH [S, T, d], dw [d]) in float64.  The
    forward is recomputed here from H and w, as under the activation
    checkpointing that wraps AttnRes in training ([Tutorial] ch. 4.6).
    The chain rule, step by step, is written out in _backward_core."""
    H = np.asarray(H, dtype=np.float64)
    c = _backward_core(H, np.asarray(w, np.float64), np.asarray(dr, np.float64), eps)
    return c["dH"], c["dw_tok"].sum(axis=0)


def backward_rounding_sites(H: np.ndarray, w: np.ndarray, dr: np.ndarray, eps: float = EPS) -> list:
    """The rounding model behind depth_attention_backward_scales: every
    quantity a straightforward evaluation of _backward_core rounds, as
    (site, index, unit) triples -- a one-unit change of quantity `site`
    [index] moves it by `unit` ([T]), one rounding's worth:
        ss_j  : sum of squares (its roundings, then rho's: 4 d rho^2)   ss_j + 4 d rho_j^2
        g_j   : dot product dr . h_j (its absolute terms)                 sum_c |dr_c h_jc|
        z_j   : w . h_j / rho_j, then z - max and its exponential (the
                dot's absolute terms mapped by 1/rho; one unit each of
                z, z - max and the exponential's relative error)        sum_c|w_c h_jc|/rho_j + |z_j| + |z_j - m| + 1
        a_j   : the sum of the exponentials and the division by it
                (relative errors that do not keep sum_j a_j = 1)        2 a_j
        gbar  : one unit per product a_k g_k                             sum_k a_k |g_k|
        dz_j  : a subtraction and a product                              2 |dz_j|
        alpha_j: a division                                              |alpha_j|
        beta_j : three operations                                        3 |beta_j|
    The final elementwise products and sums of dh and the sum of dw are
    counted in depth_attention_backward_scales itself."""
    H = np.asarray(H, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dr = np.asarray(dr, dtype=np.float64)
    S, T, d = H.shape
    c = _backward_core(H, w, dr, eps)
    absP = np.einsum("std,d->st", np.abs(H), np.abs(w))
    absG = np.einsum("std,td->st", np.abs(H), np.abs(dr))
    sites = []
    for j in range(S):
        sites.append(("ss", j, c["ss"][j] + 4 * d * c["rho"][j] ** 2))
        sites.append(("g", j, absG[j]))
        sites.append(("z", j, absP[j] / c["rho"][j] + np.abs(c["z"][j]) + np.abs(c["z"][j] - c["m"][0]) + 1))
        sites.append(("a", j, 2 * c["a"][j]))
        sites.append(("dz", j, 2 * np.abs(c["dz"][j])))
        sites.append(("alpha", j, np.abs(c["alpha"][j])))
        sites.append(("beta", j, 3 * np.abs(c["beta"][j])))
    sites.append(("gbar", 0, (c["a"] * np.abs(c["g"])).sum(axis=0)))
    return sites


_RESPOND_ARG = {"ss": "dss", "g": "dg", "z": "dz_", "a": "da_", "gbar": "dgbar", "dz": "ddz", "alpha": "dalpha",
                "beta": "dbeta"}


def backward_scalar_sensitivities(H: np.ndarray, w: np.ndarray, dr: np.ndarray,
                                  eps: float = EPS) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """First-order rounding sensitivities of the per-token scalars a_s,
    alpha_s, beta_s of _backward_core: for each,
        sum over the sites of backward_rounding_sites |d x_s / d site| * unit(site),
    the change of x_s when every rounded quantity moves by one unit of its
    own size in the worst direction.  The derivatives follow
    _backward_core step by step (chain rule, written out below).
    Returns (sens_a, sens_alpha, sens_beta), each [S, T]."""
    H = np.asarray(H, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dr = np.asarray(dr, dtype=np.float64)
    S, T, d = H.shape
    c = _backward_core(H, w, dr, eps)
    a, g, gbar, rho, z, alpha, beta = c["a"], c["g"], c["gbar"], c["rho"], c["z"], c["alpha"], c["beta"]

    def respond(dss=0.0, dg=0.0, dz_=0.0, da_=0.0, dgbar=0.0, ddz=0.0, dalpha=0.0, dbeta=0.0):
        # first-order changes of (a, alpha, beta) [S, T] for changes of the
        # intermediates
        drho = dss / (2 * d * rho)                            # rho^2 = ss/d + eps
        dzt = dz_ - z * drho / rho                            # z = p / rho
        da = a * (dzt - (a * dzt).sum(axis=0, keepdims=True)) + da_  # softmax, then its rounding
        dgb = (da * g).sum(axis=0, keepdims=True) + (a * dg).sum(axis=0, keepdims=True) + dgbar
        ddzt = da * (g - gbar) + a * (dg - dgb) + ddz
        dal = ddzt / rho - alpha * drho / rho + dalpha
        dbe = (dal * z + alpha * dzt) / (d * rho) - beta * drho / rho + dbeta
        return da, dal, dbe

    sa, sal, sbe = np.zeros((S, T)), np.zeros((S, T)), np.zeros((S, T))
    for site, j, unit in backward_rounding_sites(H, w, dr, eps):
        one = np.zeros((1 if site == "gbar" else S, T))
        one[j] = 1.0
        da, dal, dbe = respond(**{_RESPOND_ARG[site]: one})
        sa += np.abs(da) * unit
        sal += np.abs(dal) * unit
        sbe += np.abs(dbe) * unit
    return sa, sal, sbe


def depth_attention_backward_scales(H: np.ndarray, w: np.ndarray, dr: np.ndarray,
                                    eps: float = EPS) -> tuple[np.ndarray, np.ndarray]:
    """Condition scales of the two gradients, for tolerances: how far an
    evaluation moves each output when every rounded quantity moves by one
    unit of its own size (backward_rounding_sites), to first order and all
    in the worst direction.  With the scalar sensitivities of
    backward_scalar_sensitivities (sens_*) and one unit each for the final
    products and sums,
        dH_scale[s, t, c] = (sens_a + 2|a_s|) |dr_c| + (sens_alpha + 2|alpha_s|) |w_c|
                            + (sens_beta + 2|beta_s|) |h_sc|
        dw_scale[c]       = sum_t sum_s (sens_alpha + 2|alpha_s|) |h_sc|
    (every term of dh = a dr + alpha w - beta h and of dw = sum alpha h
    counted with its absolute value).  Returns (dH_scale [S, T, d],
    dw_scale [d]).  An evaluation with unit roundoff u errs by about u
    times the scale or less: rounding errors of opposite sign cancel, and
    the sum over tokens of dw is counted as if all its errors had one
    sign."""
    H = np.asarray(H, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dr = np.asarray(dr, dtype=np.float64)
    c = _backward_core(H, w, dr, eps)
    sa, sal, sbe = backward_scalar_sensitivities(H, w, dr, eps)
    A = sa + 2 * np.abs(c["a"])
    B = sal + 2 * np.abs(c["alpha"])
    C = sbe + 2 * np.abs(c["beta"])
    dHs = A[:, :, None] * np.abs(dr)[None] + B[:, :, None] * np.abs(w)[None, None, :] + C[:, :, None] * np.abs(H)
    dws = np.einsum("st,std->d", B, np.abs(H))
    return dHs, dws


# --------------------------------------------------------------------------
# Block bookkeeping: which sources layer l sees   [Tutorial ch. 4.3 Eq. 10]
# --------------------------------------------------------------------------

def block_index(layer: int, block_size: int) -> int:
    """Block n (1-based) that layer `layer` (1-based) belongs to."""
    return (layer - 1) // block_size + 1


def position_in_block(layer: int, block_size: int) -> int:
    """Position i (1-based) of layer `layer` inside its block."""
    return (layer - 1) % block_size + 1


def num_blocks(num_layers: int, block_size: int) -> int:
    """N = ceil(L / B); the last block may be incomplete ([Tutorial ch. 4.5])."""
    return -(-num_layers // block_size)


def block_layers(n: int, block_size: int, num_layers: int) -> range:
    """The layers whose outputs are summed into block representation b_n."""
    first = (n - 1) * block_size + 1
    last = min(n * block_size, num_layers)
    return range(first, last + 1)


def value_list(layer: int, block_size: int, num_layers: int) -> list[tuple]:
    """Eq. 10's value list for `layer` in 1..L, or the final output for L+1.

    Entries, in source order:
      ("embed",)                      b_0 = h_0, the token embedding
      ("block", k, first, last)       b_k = sum of outputs of layers first..last
      ("partial", n, first, last)     the current block's partial sum over
                                      layers first..last (only when non-empty:
                                      the block's first layer gets no zero
                                      source)
    [Tutorial ch. 4.3]: layer i of block n reads [b_0 .. b_{n-1}] when i = 1
    and [b_0 .. b_{n-1}, b_n^{i-1}] when i >= 2; the final output layer reads
    all N block representations ([Tutorial ch. 4.3], last paragraph).
    """
    L, B = num_layers, block_size
    if not (1 <= layer <= L + 1):
        raise ValueError("layer out of range")
    out: list[tuple] = [("embed",)]
    if layer == L + 1:
        for k in range(1, num_blocks(L, B) + 1):
            lay = block_layers(k, B, L)
            out.append(("block", k, lay[0], lay[-1]))
        return out
    n, i = block_index(layer, B), position_in_block(layer, B)
    for k in range(1, n):
        lay = block_layers(k, B, L)
        out.append(("block", k, lay[0], lay[-1]))
    if i >= 2:
        first = (n - 1) * B + 1
        out.append(("partial", n, first, layer - 1))
    return out


def num_sources(layer: int, block_size: int, num_layers: int) -> int:
    """Number of sources layer `layer` attends over (len of the value list)."""
    return len(value_list(layer, block_size, num_layers))


# --------------------------------------------------------------------------
# Storage rounding (the stack stores every tensor it writes in bf16 or fp32)
# --------------------------------------------------------------------------

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even,
    returned as float64.  bfloat16 keeps 8 significant bits and fp32's
    exponent range (subnormal quantum 2^-133); overflow gives +-inf."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = m 2^e, 0.5 <= |m| < 1
    q = np.maximum(e - 8, -133)              # quantum exponent of x's binade
    y = np.ldexp(np.rint(np.ldexp(x, -q)), q)  # rint: round half to even
    return np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, x), y)


def round_fp32(x: np.ndarray) -> np.ndarray:
    """Round float64 values to float32 (IEEE, ties to even), returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _identity(x):
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# The synthetic layer body that stands in for KDA/MLA + MoE in the stack
# --------------------------------------------------------------------------

def synthetic_layer(x: np.ndarray, g: np.ndarray, s: np.ndarray) -> np.ndarray:
    """F_l(x) = tanh(x * g_l) * s_l, per channel (a stand-in layer body, not
    part of the method)."""
    x = np.asarray(x, dtype=np.float64)
    return np.tanh(x * np.asarray(g, np.float64)) * np.asarray(s, np.float64)


def synthetic_layer_backward(x: np.ndarray, g: np.ndarray, s: np.ndarray, dv: np.ndarray) -> np.ndarray:
    """Gradient through F_l: d/dx [tanh(x g) s] = (1 - tanh(x g)^2) g s, times
    the incoming gradient dv (per channel; the stand-in body, not the method)."""
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(g, np.float64)
    th = np.tanh(x * g)
    return np.asarray(dv, np.float64) * (1.0 - th * th) * g * np.asarray(s, np.float64)


# --------------------------------------------------------------------------
# Stacks
# --------------------------------------------------------------------------

@dataclass
class StackTrace:
    """Everything a stack forward produced, per layer (index 0 = layer 1)."""
    r: list = field(default_factory=list)          # r_l [T, d], l = 1..L+1 (as stored)
    a: list = field(default_factory=list)          # a_l [T, S_l], l = 1..L+1
    v: list = field(default_factory=list)          # v_l = F_l(r_l) [T, d], l = 1..L (as stored)
    final_sources: list = field(default_factory=list)  # sources of the final aggregation


def _range_sum(outputs: dict, first: int, last: int, store: Callable, memo: dict) -> np.ndarray:
    """Sum of the layer outputs v_first .. v_last, added in layer order with
    every running total stored (rounded) once:
        ((v_first + v_{first+1}) -> store) + v_{first+2} -> store ...
    (a plain sum when `store` is exact).  Memoised per range: the sum over
    first..last is the stored sum over first..last-1 plus v_last."""
    key = (first, last)
    if key not in memo:
        if last == first:
            memo[key] = outputs[first]
        else:
            memo[key] = store(_range_sum(outputs, first, last - 1, store, memo) + outputs[last])
    return memo[key]


def block_stack_forward(h0: np.ndarray, W: np.ndarray, layer_fn: Callable[[int, np.ndarray], np.ndarray],
                        num_layers: int, block_size: int, eps: float = EPS,
                        store: Callable | None = None) -> StackTrace:
    """Block AttnRes forward through L layers and the final aggregation.

    Layer l (1..L) aggregates the sources of `value_list(l)` with pseudo-query
    W[l-1], giving r_l; the layer body then gives v_l = layer_fn(l, r_l), the
    layer's OUTPUT (not r_l + v_l: keys and values are the layer outputs,
    [Tutorial ch. 4.2], and b_n is the sum of the outputs of block n,
    [Tutorial ch. 4.3]).  After layer L the final aggregation (l = L+1) uses
    W[L] over [h_0, b_1 .. b_N].

    Every source is looked up from the list of layer outputs for each layer
    (b_k and the partial sum are sums over explicit layer ranges).  `store`
    models storage rounding (e.g. `round_bf16`): it is applied to every
    tensor the stack writes (r_l, v_l, and each running total of a block sum);
    None means exact fp64 throughout.
    """
    store = store or _identity
    L, B = num_layers, block_size
    W = np.asarray(W, dtype=np.float64)
    h0 = np.asarray(h0, dtype=np.float64)
    outputs = {0: h0}                               # v_0 = h_0
    memo: dict = {}
    tr = StackTrace()
    for layer in range(1, L + 2):
        srcs = []
        for entry in value_list(layer, B, L):
            if entry[0] == "embed":
                srcs.append(h0)
            else:
                _, _, first, last = entry
                srcs.append(_range_sum(outputs, first, last, store, memo))
        r, a = depth_attention(np.stack(srcs), W[layer - 1], eps)
        r = store(r)
        tr.r.append(r)
        tr.a.append(a)
        if layer <= L:
            v = store(layer_fn(layer, r))
            outputs[layer] = v
            tr.v.append(v)
        else:
            tr.final_sources = srcs
    return tr


def full_stack_forward(h0: np.ndarray, W: np.ndarray, layer_fn: Callable[[int, np.ndarray], np.ndarray],
                       num_layers: int, eps: float = EPS) -> StackTrace:
    """Full AttnRes: layer l attends over [h_0, v_1 .. v_{l-1}] (every earlier
    layer output, [Deep-dive 2 §2] H_<l; [Tutorial ch. 4.2]); the final output
    over [h_0, v_1 .. v_L].  Exact fp64; written separately from the block
    version so the two can check each other."""
    W = np.asarray(W, dtype=np.float64)
    history = [np.asarray(h0, dtype=np.float64)]
    tr = StackTrace()
    for layer in range(1, num_layers + 2):
        r, a = depth_attention(np.stack(history), W[layer - 1], eps)
        tr.r.append(r)
        tr.a.append(a)
        if layer <= num_layers:
            v = np.asarray(layer_fn(layer, r), dtype=np.float64)
            tr.v.append(v)
            history.append(v)
        else:
            tr.final_sources = list(history)
    return tr


def block_stack_backward(h0: np.ndarray, W: np.ndarray, G: np.ndarray, Sc: np.ndarray,
                         num_layers: int, block_size: int, dr_out: np.ndarray,
                         eps: float = EPS) -> tuple[np.ndarray, np.ndarray]:
    """Gradients of the loss sum(r_{L+1} * dr_out) of a Block AttnRes stack
    whose layer bodies are synthetic_layer(., G[l-1], Sc[l-1]), with respect
    to the embedding h_0 and the pseudo-queries W[0..L].  Exact fp64.

    Reverse mode over the value lists ([Tutorial ch. 4.3] Eq. 10): every
    source of layer l is h_0 or a sum of layer outputs v_first..v_last, so the
    gradient layer l's aggregation sends to that source reaches each of those
    outputs unchanged.  Layers are visited from the final aggregation down to
    layer 1; when layer j is reached every layer that reads v_j (later layers
    of its block through the partial sum, later blocks and the final
    aggregation through b_n) has been visited, so dL/dv_j is complete and
    goes through the layer body to r_j, dL/dr_j = dL/dv_j F_j'(r_j), and on
    into layer j's own aggregation.  The forward is recomputed from h_0, W,
    G, Sc (as under activation checkpointing, [Tutorial] ch. 4.6).
    Returns (dh0 [T, d], dW [L+1, d]).
    """
    L, B = num_layers, block_size
    G = np.asarray(G, np.float64)
    Sc = np.asarray(Sc, np.float64)
    fn = lambda l, x: synthetic_layer(x, G[l - 1], Sc[l - 1])
    tr = block_stack_forward(h0, W, fn, L, B, eps)
    v = {0: np.asarray(h0, np.float64)}
    for j in range(1, L + 1):
        v[j] = tr.v[j - 1]
    dv = {j: np.zeros_like(v[0]) for j in range(0, L + 1)}
    dW = np.zeros((L + 1, v[0].shape[1]))
    for layer in range(L + 1, 0, -1):
        if layer == L + 1:
            dr = np.asarray(dr_out, np.float64)
        else:
            dr = synthetic_layer_backward(tr.r[layer - 1], G[layer - 1], Sc[layer - 1], dv[layer])
        entries = value_list(layer, B, L)
        srcs = []
        for entry in entries:
            if entry[0] == "embed":
                srcs.append(v[0])
            else:
                _, _, first, last = entry
                srcs.append(sum(v[j] for j in range(first, last + 1)))
        dH, dW[layer - 1] = depth_attention_backward(np.stack(srcs), W[layer - 1], dr, eps)
        for entry, dh in zip(entries, dH):
            if entry[0] == "embed":
                dv[0] += dh
            else:
                _, _, first, last = entry
                for j in range(first, last + 1):
                    dv[j] += dh
    return dv[0], dW
