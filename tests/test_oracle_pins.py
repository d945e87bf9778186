"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Each test is chosen so that a plausible mistake in the oracle (a dropped
term, a wrong axis, a transposed operand, eps in the wrong place, a 1/sqrt(d)
temperature, normalised values instead of raw ones, an off-by-one in the
block bookkeeping) fails at least one of them.  None of them calls the CUDA
path.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from tests.conftest import read_golden

RNG = np.random.default_rng(12345)


# ---------------------------------------------------------------- helpers ---

def _orth_to(w, y):
    """Component of y orthogonal to w."""
    return y - (y @ w) / (w @ w) * w


def _sources_with_logits(w, z, d, T=1, eps=O.EPS, ms=1.0, rng=RNG):
    """Sources h_s (s = 0..S-1) whose RMSNorm logits against w are exactly z_s.

    h_s = c_s u + y_s with u = w / |w|^2 (so w.h_s = c_s) and y_s orthogonal
    to w, scaled so that mean(h_s^2) = ms; then rms = sqrt(ms + eps) and
    choosing c_s = z_s sqrt(ms + eps) gives logit z_s.
    """
    u = w / (w @ w)
    H = np.empty((len(z), T, d))
    for s, zs in enumerate(z):
        c = zs * math.sqrt(ms + eps)
        for t in range(T):
            y = _orth_to(w, rng.standard_normal(d))
            need = d * ms - c * c * (u @ u)
            assert need > 0
            y *= math.sqrt(need / (y @ y))
            H[s, t] = c * u + y
    return H


# ------------------------------------------------- worked example (§2.1) ---

def test_worked_example_four_sources(golden_dir):
    rows = read_golden(os.path.join(golden_dir, "worked_example_4src.txt"))
    a_page = np.array([float(r[1]) for r in rows])
    assert [int(r[0]) for r in rows] == [0, 1, 2, 3]
    assert abs(a_page.sum() - 1.0) < 1e-15
    d = 256
    w = RNG.standard_normal(d) / math.sqrt(d)
    H = _sources_with_logits(w, np.log(a_page), d, T=3)
    r, a = O.depth_attention(H, w)
    np.testing.assert_allclose(a, np.tile(a_page, (3, 1)), rtol=0, atol=1e-12)
    # r_4 = 0.05 h_0 + 0.10 h_1 + 0.70 h_2 + 0.15 h_3, from the page's weights
    r_page = 0.05 * H[0] + 0.10 * H[1] + 0.70 * H[2] + 0.15 * H[3]
    np.testing.assert_allclose(r, r_page, rtol=1e-12, atol=1e-12 * np.abs(H).max())


# ------------------------------------------------ definitions & closed forms -

def test_rms_closed_form_constant_rows():
    # a constant row c*1 has mean square c^2; eps goes inside the root
    for c in [0.0, 1e-3, 0.5, -2.0, 37.0]:
        for eps in [0.0, 1e-5, 0.25]:
            h = np.full((1, 64), c)
            assert abs(O.rms(h, eps)[0] - math.sqrt(c * c + eps)) <= 1e-15 * max(1, abs(c))
    # mean over the channel axis, not over tokens: rows with different scales
    h = np.stack([np.full(16, 1.0), np.full(16, 3.0)])
    np.testing.assert_allclose(O.rms(h, 0.0), [1.0, 3.0], rtol=1e-15)


def test_logits_closed_form_constant_sources():
    # h_s[t] = c_{s,t} * 1 (all channels equal): logit = c sum(w) / sqrt(c^2 + eps),
    # with no 1/sqrt(d) temperature; weights follow.
    d, S, T = 48, 3, 5
    w = RNG.standard_normal(d)
    c = RNG.uniform(-3, 3, size=(S, T))
    H = np.repeat(c[:, :, None], d, axis=2)
    for eps in [0.0, 1e-5, 0.5]:
        z = (c * w.sum() / np.sqrt(c * c + eps)).T          # [T, S]
        a_cf = np.exp(z - z.max(1, keepdims=True))
        a_cf /= a_cf.sum(1, keepdims=True)
        r_cf = (a_cf * c.T).sum(1)                          # every channel of r equals this
        r, a = O.depth_attention(H, w, eps)
        np.testing.assert_allclose(a, a_cf, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(r, np.repeat(r_cf[:, None], d, 1), rtol=1e-13, atol=1e-15)


def test_single_source_returns_it_exactly():
    # layer 1 of a block stack sees only h_0: weight 1, r = h_0 bit for bit
    h = RNG.standard_normal((1, 7, 33))
    r, a = O.depth_attention(h, RNG.standard_normal(33))
    assert np.array_equal(a, np.ones((7, 1)))
    assert np.array_equal(r, h[0])


def test_zero_query_is_uniform_mean():
    # uniform mixer: zero logits -> w_i = 1/N -> output = sum_i source_i / N
    S, T, d = 5, 4, 24
    H = RNG.standard_normal((S, T, d)) * RNG.uniform(0.1, 10, size=(S, 1, 1))
    r, a = O.depth_attention(H, np.zeros(d))
    np.testing.assert_allclose(a, np.full((T, S), 1.0 / S), rtol=1e-15)
    np.testing.assert_allclose(r, H.mean(0), rtol=1e-13, atol=1e-14)


def test_dominant_logit_selects_that_source():
    d = 128
    w = RNG.standard_normal(d)          # |w|^2 ~ d leaves room for logit 45
    for j in range(4):
        z = np.zeros(4)
        z[j] = 45.0                          # other weights ~ e^-45 ~ 3e-20
        H = _sources_with_logits(w, z, d, T=2)
        r, a = O.depth_attention(H, w)
        np.testing.assert_allclose(a[:, j], 1.0, rtol=0, atol=1e-15)
        np.testing.assert_allclose(r, H[j], rtol=0, atol=1e-15 * np.abs(H).max() * 8)


def test_values_are_raw_sources_not_normalised():
    # scaling a source by k keeps its weight (with eps = 0) but scales its
    # contribution to r by k: values are the un-normalised sources
    d, S, T = 32, 3, 4
    H = RNG.standard_normal((S, T, d))
    w = RNG.standard_normal(d) / math.sqrt(d)
    r0, a0 = O.depth_attention(H, w, eps=0.0)
    H2 = H.copy()
    H2[1] *= 7.0
    r1, a1 = O.depth_attention(H2, w, eps=0.0)
    np.testing.assert_allclose(a1, a0, rtol=1e-13)
    np.testing.assert_allclose(r1 - r0, 6.0 * a0[:, 1:2] * H[1], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- invariants ---

def test_weights_nonnegative_sum_to_one_and_convex_hull():
    for S in [1, 2, 4, 9, 17]:
        H = RNG.standard_normal((S, 6, 40)) * RNG.uniform(0.01, 100, size=(S, 6, 1))
        w = RNG.standard_normal(40) * 0.5
        r, a = O.depth_attention(H, w)
        assert (a >= 0).all()
        np.testing.assert_allclose(a.sum(1), 1.0, rtol=0, atol=1e-15)
        lo, hi = H.min(0), H.max(0)
        tol = 1e-13 * np.abs(H).max()
        assert (r >= lo - tol).all() and (r <= hi + tol).all()


def test_permuting_sources_permutes_weights_keeps_output():
    S, T, d = 6, 5, 20
    H = RNG.standard_normal((S, T, d))
    w = RNG.standard_normal(d)
    r, a = O.depth_attention(H, w)
    perm = RNG.permutation(S)
    rp, ap = O.depth_attention(H[perm], w)
    np.testing.assert_allclose(ap, a[:, perm], rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(rp, r, rtol=1e-13, atol=1e-14)


def test_rescaling_one_source_leaves_weights_unchanged():
    # the purpose of the RMSNorm keys: a large-norm source cannot dominate
    # merely by its norm.  Exact at eps = 0; with eps > 0 the change is tiny
    # but not zero (eps is really used).
    S, T, d = 4, 3, 64
    H = RNG.standard_normal((S, T, d))
    w = RNG.standard_normal(d) / math.sqrt(d)
    _, a0 = O.depth_attention(H, w, eps=0.0)
    for k in [1e-3, 0.5, 3.0, 1e4]:
        H2 = H.copy()
        H2[2] *= k
        _, a1 = O.depth_attention(H2, w, eps=0.0)
        np.testing.assert_allclose(a1, a0, rtol=1e-13, atol=1e-16)
    _, a_eps = O.depth_attention(H, w, eps=1e-5)
    H2 = H.copy()
    H2[2] *= 1e-2                      # mean square 1e-4: eps now matters (~5%)
    _, a_eps2 = O.depth_attention(H2, w, eps=1e-5)
    diff = np.abs(a_eps2 - a_eps).max()
    assert 1e-6 < diff < 0.1


# -------------------------------------------------------- bf16 rounding pin -

def test_round_bf16_matches_torch_on_fp32_values():
    x = np.concatenate([
        RNG.standard_normal(20000) * 10.0 ** RNG.integers(-30, 30, 20000),
        RNG.standard_normal(2000),
        [0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1e-40, -1e-42],
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: rounds to 1 (even)
    assert O.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: rounds up (even)
    assert O.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    # just above a tie rounds away
    assert O.round_bf16(np.array([1 + 2 ** -8 + 2 ** -40]))[0] == 1 + 2 ** -7
    assert O.round_bf16(np.array([-(1 + 2 ** -8 + 2 ** -40)]))[0] == -(1 + 2 ** -7)


# ------------------------------------------------ block bookkeeping (Eq. 10) -

def test_k3_block_layout_and_source_counts(golden_dir):
    g = {r[0]: int(r[1]) for r in read_golden(os.path.join(golden_dir, "k3_block_layout.txt"))}
    L, B = g["num_layers"], g["block_size"]
    assert O.num_blocks(L, B) == g["num_blocks"]
    assert len(O.block_layers(g["num_blocks"], B, L)) == g["last_block_layers"]
    assert list(O.block_layers(8, B, L)) == list(range(85, 94))
    counts = [O.num_sources(l, B, L) for l in range(1, L + 2)]
    # the final aggregation sees the embedding plus all 8 block representations
    assert counts[-1] == g["block_sources"] == math.ceil(L / B) + 1
    assert max(counts) == g["block_sources"]
    # Full AttnRes (block size 1): L outputs + embedding at the top
    assert O.num_sources(L + 1, 1, L) == g["full_sources"] == L + 1
    # derived totals: 12n + 11 per full block n = 1..7, 8*9 + 8 for the last
    assert sum(counts[:L]) == 493
    assert counts[0] == 1 and counts[1] == 2 and counts[11] == 2
    assert counts[12] == 2 and counts[13] == 3          # layer 13 opens block 2
    assert counts[84] == 8 and counts[85] == 9           # layer 85 opens block 8
    # the site's per-token state estimate
    d = g["hidden"]
    assert abs(L * d - g["full_values_per_token_approx"]) / g["full_values_per_token_approx"] < 0.01
    assert abs(9 * d - g["block_values_per_token_approx"]) / g["block_values_per_token_approx"] < 0.01
    assert abs(L * d * 2 / 1e6 - 1.3) < 0.05 and abs(9 * d * 2 / 1e3 - 129) < 1


def test_value_list_two_cases():
    L, B = 93, 12
    # first layer of block 3: [b_0, b_1, b_2], no empty partial
    assert O.value_list(25, B, L) == [("embed",), ("block", 1, 1, 12), ("block", 2, 13, 24)]
    # layer 3 of block 3: ... plus the partial sum of layers 25, 26
    assert O.value_list(27, B, L)[-1] == ("partial", 3, 25, 26)
    # final output: embedding plus the 8 blocks, the last one layers 85..93
    fin = O.value_list(94, B, L)
    assert fin[0] == ("embed",) and fin[-1] == ("block", 8, 85, 93) and len(fin) == 9
    # block size 1 is Full AttnRes: layer l sees the embedding and l-1 outputs
    for l in range(1, 8):
        vl = O.value_list(l, 1, 7)
        assert vl == [("embed",)] + [("block", k, k, k) for k in range(1, l)]
    with pytest.raises(ValueError):
        O.value_list(0, B, L)
    with pytest.raises(ValueError):
        O.value_list(L + 2, B, L)


# --------------------------------------------------------- synthetic layer --

def test_synthetic_layer_closed_forms():
    g = np.array([2.0, -0.5, 1.0])
    s = np.array([0.1, 0.2, 0.05])
    assert np.array_equal(O.synthetic_layer(np.zeros(3), g, s), np.zeros(3))
    x = np.arctanh(0.5) / g                      # tanh(x g) = 0.5
    np.testing.assert_allclose(O.synthetic_layer(x, g, s), 0.5 * s, rtol=1e-15)
    np.testing.assert_allclose(O.synthetic_layer(-x, g, s), -0.5 * s, rtol=1e-15)


# ---------------------------------------------------------------- stacks ----

def _tiny_stack(L, d, T, seed):
    rng = np.random.default_rng(seed)
    h0 = rng.standard_normal((T, d))
    W = rng.standard_normal((L + 1, d)) / math.sqrt(d)
    G = rng.standard_normal((L, d))
    Sc = rng.uniform(0.05, 0.2, size=(L, d))
    fn = lambda l, x: O.synthetic_layer(x, G[l - 1], Sc[l - 1])
    return h0, W, G, Sc, fn


def test_block_size_one_equals_full_attnres():
    L, d, T = 6, 16, 3
    h0, W, G, Sc, fn = _tiny_stack(L, d, T, 7)
    blk = O.block_stack_forward(h0, W, fn, L, 1)
    full = O.full_stack_forward(h0, W, fn, L)
    for l in range(L + 1):
        np.testing.assert_allclose(blk.a[l], full.a[l], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(blk.r[l], full.r[l], rtol=1e-13, atol=1e-14)
    for s_b, s_f in zip(blk.final_sources, full.final_sources):
        np.testing.assert_allclose(s_b, s_f, rtol=1e-13, atol=1e-14)


def test_block_size_at_least_L_is_embedding_plus_partial():
    # one block holding every layer: layer l >= 2 sees [h_0, v_1 + .. + v_{l-1}]
    L, d, T = 5, 12, 2
    h0, W, G, Sc, fn = _tiny_stack(L, d, T, 8)
    tr = O.block_stack_forward(h0, W, fn, L, L)
    for l in range(2, L + 1):
        part = sum(tr.v[j - 1] for j in range(1, l))
        r, a = O.depth_attention(np.stack([h0, part]), W[l - 1])
        np.testing.assert_allclose(tr.r[l - 1], r, rtol=1e-13, atol=1e-14)
    assert len(tr.final_sources) == 2
    np.testing.assert_allclose(tr.final_sources[1], sum(tr.v), rtol=1e-13, atol=1e-14)


def test_stack_rounding_mode_stores_bf16_values():
    L, d, T = 7, 16, 3
    h0, W, G, Sc, fn = _tiny_stack(L, d, T, 9)
    h0 = O.round_bf16(h0)
    tr = O.block_stack_forward(h0, W, fn, L, 3, store=O.round_bf16)
    for x in tr.r + tr.v + tr.final_sources:
        assert np.array_equal(O.round_bf16(x), x)
    ex = O.block_stack_forward(h0, W, fn, L, 3)
    # rounding only perturbs at the bf16 level
    np.testing.assert_allclose(tr.r[-1], ex.r[-1], rtol=0.05, atol=0.05)


def _running_state_stack(h0, W, G, Sc, L, B, store, slip=None):
    """A second, independent statement of a stack with storage rounding,
    written as the running state a stack keeps (Eq. 10's two cases): the
    stored values are rounded exactly where they are written -- r_l, the
    layer output v_l, and every new partial sum or block sum (the fp64 sum
    of the stored partial sum and v_l, rounded once).  `slip` plants one of
    three plausible misplacements of the rounding (to show the pin sees
    them): "block_only" rounds a block sum only when it is finished,
    "raw_r" feeds the layer body the unrounded r_l, "late_v" adds the
    unrounded v_l and rounds it afterwards."""
    blocks, partial, exact_partial = [], None, None
    rs, as_, vs = [], [], []
    for layer in range(1, L + 2):
        srcs = [h0] + blocks + ([partial] if partial is not None else [])
        r_raw, a = O.depth_attention(np.stack(srcs), W[layer - 1])
        r = store(r_raw)
        rs.append(r)
        as_.append(a)
        if layer == L + 1:
            return rs, as_, vs, srcs
        v_raw = O.synthetic_layer(r_raw if slip == "raw_r" else r, G[layer - 1], Sc[layer - 1])
        v = store(v_raw)
        vs.append(v)
        add = v_raw if slip == "late_v" else v
        if slip == "block_only":
            exact_partial = add if exact_partial is None else exact_partial + add
            partial = exact_partial
        else:
            partial = add if partial is None else store(partial + add)
            if slip == "late_v":
                partial = store(partial)
        if layer % B == 0 or layer == L:      # the block ends here
            blocks.append(store(partial))
            partial, exact_partial = None, None


@pytest.mark.parametrize("B", [1, 2, 3])
@pytest.mark.parametrize("L", [1, 4, 7])
def test_storage_rounding_is_placed_at_every_store(L, B):
    # c12: with bf16 storage the oracle rounds r_l, v_l and each new partial
    # or block sum once, where a stack stores them; checked bit for bit
    # against the running-state statement above (fp64 between the stores)
    h0, W, G, Sc, _ = _tiny_stack(L, 8, 3, 200 + 10 * L + B)
    h0 = O.round_bf16(h0)
    fn = lambda l, x: O.synthetic_layer(x, G[l - 1], Sc[l - 1])
    tr = O.block_stack_forward(h0, W, fn, L, B, store=O.round_bf16)
    rs, as_, vs, final = _running_state_stack(h0, W, G, Sc, L, B, O.round_bf16)
    for l in range(L + 1):
        assert np.array_equal(tr.r[l], rs[l]) and np.array_equal(tr.a[l], as_[l]), f"layer {l + 1}"
    for l in range(L):
        assert np.array_equal(tr.v[l], vs[l]), f"v_{l + 1}"
    assert len(tr.final_sources) == len(final)
    for x, y in zip(tr.final_sources, final):
        assert np.array_equal(x, y)


def test_storage_rounding_pin_sees_misplaced_roundings():
    # the three slips of the running-state statement each change some stored
    # value of a 7-layer stack with blocks of 3 (so the pin above would fail
    # for an oracle that made one of them)
    L, B = 7, 3
    h0, W, G, Sc, _ = _tiny_stack(L, 8, 3, 290)
    h0 = O.round_bf16(h0)
    ref = _running_state_stack(h0, W, G, Sc, L, B, O.round_bf16)
    for slip in ("block_only", "raw_r", "late_v"):
        got = _running_state_stack(h0, W, G, Sc, L, B, O.round_bf16, slip=slip)
        same = all(np.array_equal(x, y) for x, y in zip(ref[0] + ref[2] + ref[3], got[0] + got[2] + got[3]))
        assert not same, slip


def test_round_fp32_ties_to_even():
    # 1 + 2^-24 is halfway between 1 and 1 + 2^-23: rounds to 1 (even);
    # 1 + 3*2^-24 is halfway between 1 + 2^-23 and 1 + 2^-22: rounds up (even)
    x = np.array([1 + 2 ** -24, 1 + 3 * 2 ** -24, -(1 + 3 * 2 ** -24), 1 + 2 ** -24 + 2 ** -50, 2.0 ** -149 * 0.5])
    want = np.array([1.0, 1 + 2 ** -22, -(1 + 2 ** -22), 1 + 2 ** -23, 0.0])
    assert np.array_equal(O.round_fp32(x), want)


def _brute_force_stack(h0, W, G, Sc, L, B, eps=O.EPS):
    """Independent high-precision stack, written as a running-state machine
    from the two cases of Eq. 10 (the oracle instead rebuilds every source
    from explicit layer ranges).  mpmath at 40 digits, one token at a time."""
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 40
    T, d = h0.shape
    out_r, out_a = [], []
    for t in range(T):
        emb = [mp.mpf(float(x)) for x in h0[t]]
        blocks = []              # completed block representations
        partial = None           # running sum of the current block, None if empty
        rs, as_ = [], []
        for layer in range(1, L + 2):
            srcs = [emb] + blocks + ([partial] if partial is not None else [])
            wq = [mp.mpf(float(x)) for x in W[layer - 1]]
            z = []
            for h in srcs:
                ms = mp.fsum(x * x for x in h) / d
                z.append(mp.fsum(a * b for a, b in zip(wq, h)) / mp.sqrt(ms + mp.mpf(eps)))
            m = max(z)
            e = [mp.exp(zz - m) for zz in z]
            tot = mp.fsum(e)
            a = [ee / tot for ee in e]
            r = [mp.fsum(a[s] * srcs[s][c] for s in range(len(srcs))) for c in range(d)]
            rs.append([float(x) for x in r])
            as_.append([float(x) for x in a])
            if layer == L + 1:
                break
            v = [mp.tanh(r[c] * mp.mpf(float(G[layer - 1, c]))) * mp.mpf(float(Sc[layer - 1, c]))
                 for c in range(d)]
            partial = v if partial is None else [p + q for p, q in zip(partial, v)]
            if layer % B == 0 or layer == L:      # the block ends here
                blocks.append(partial)
                partial = None
        out_r.append(rs)
        out_a.append(as_)
    return out_r, out_a


@pytest.mark.parametrize("L,B", [(4, 1), (5, 2), (7, 3), (6, 3), (7, 2)])
def test_block_stack_matches_brute_force(L, B):
    d, T = 8, 2
    h0, W, G, Sc, fn = _tiny_stack(L, d, T, 100 + 10 * L + B)
    tr = O.block_stack_forward(h0, W, fn, L, B)
    br, ba = _brute_force_stack(h0, W, G, Sc, L, B)
    for l in range(L + 1):
        for t in range(T):
            np.testing.assert_allclose(tr.r[l][t], br[t][l], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(tr.a[l][t], ba[t][l], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------- backward -----

def _loss(H, w, dr, eps):
    r, _ = O.depth_attention(H, w, eps)
    return float((r * dr).sum())


@pytest.mark.parametrize("S,eps", [(1, 1e-5), (3, 1e-5), (9, 1e-5), (4, 0.0), (5, 0.3)])
def test_backward_matches_central_differences(S, eps):
    # the gradient of L = sum(dr * r) by central differences in fp64, entry by
    # entry on a sample of coordinates (independent of the analytic formulas)
    rng = np.random.default_rng(S * 7 + 1)
    T, d = 3, 24
    H = rng.standard_normal((S, T, d)) * rng.uniform(0.2, 3, size=(S, 1, 1))
    w = rng.standard_normal(d) / math.sqrt(d) * 3
    dr = rng.standard_normal((T, d))
    dH, dw = O.depth_attention_backward(H, w, dr, eps)
    step = 1e-6
    for _ in range(40):
        s, t, c = rng.integers(S), rng.integers(T), rng.integers(d)
        Hp, Hm = H.copy(), H.copy()
        Hp[s, t, c] += step
        Hm[s, t, c] -= step
        fd = (_loss(Hp, w, dr, eps) - _loss(Hm, w, dr, eps)) / (2 * step)
        assert abs(fd - dH[s, t, c]) <= 1e-7 * (1 + abs(fd)), (s, t, c, fd, dH[s, t, c])
    for c in range(d):
        wp, wm = w.copy(), w.copy()
        wp[c] += step
        wm[c] -= step
        fd = (_loss(H, wp, dr, eps) - _loss(H, wm, dr, eps)) / (2 * step)
        assert abs(fd - dw[c]) <= 1e-7 * (1 + abs(fd)), (c, fd, dw[c])


def test_backward_closed_forms():
    rng = np.random.default_rng(5)
    T, d = 4, 16
    # one source: r = h_0, so dh_0 = dr and w has no influence
    H = rng.standard_normal((1, T, d))
    dr = rng.standard_normal((T, d))
    dH, dw = O.depth_attention_backward(H, rng.standard_normal(d), dr)
    assert np.array_equal(dH[0], dr) and np.array_equal(dw, np.zeros(d))
    # zero query: uniform weights, dh_s = dr / S exactly in exact arithmetic
    S = 5
    H = rng.standard_normal((S, T, d)) * rng.uniform(0.1, 10, size=(S, 1, 1))
    dH, dw = O.depth_attention_backward(H, np.zeros(d), dr)
    np.testing.assert_allclose(dH, np.broadcast_to(dr / S, dH.shape), rtol=1e-14, atol=1e-15)
    # eps = 0: the logit is invariant to scaling h_s, so its gradient is
    # orthogonal to h_s and dh_s . h_s = a_s (dr . h_s)
    w = rng.standard_normal(d) / math.sqrt(d)
    dH, _ = O.depth_attention_backward(H, w, dr, eps=0.0)
    _, a = O.depth_attention(H, w, eps=0.0)
    lhs = np.einsum("std,std->st", dH, H)
    rhs = a.T * np.einsum("std,td->st", H, dr)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


# ------------------------------------------ backward tolerance scales -----
#
# depth_attention_backward_scales sets every backward parity bar.  It is the
# first-order worst-case change of each gradient when each rounded quantity
# of the evaluation moves by one unit of its own size.  Pinned here by
# (1) the rounding model restated from its definition, (2) every scalar
# sensitivity against central differences of the evaluation, (3) the closed
# form at S = 1, (4) an actual fp32 evaluation erring within a few units of
# it (and not far below), and (5) planted mistakes in the gradient formula
# landing far outside 1e-5 of it.

U32 = 2.0 ** -24


def _bwd_case(S, T, d, eps, qscale, seed):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((S, T, d)) * rng.uniform(0.2, 3, size=(S, 1, 1))
    w = rng.standard_normal(d) / math.sqrt(d) * qscale
    dr = rng.standard_normal((T, d))
    return H, w, dr


def _model_units(H, w, dr, eps):
    """The rounding model, restated: one unit per rounded quantity."""
    S, T, d = H.shape
    ss = (H * H).sum(axis=2)
    rho = np.sqrt(ss / d + eps)
    z = (H @ w) / rho
    e = np.exp(z - z.max(axis=0))
    a = e / e.sum(axis=0)
    g = np.einsum("std,td->st", H, dr)
    gbar = (a * g).sum(axis=0)
    dz = a * (g - gbar)
    alpha = dz / rho
    beta = alpha * z / (d * rho)
    P = np.abs(H) @ np.abs(w)
    G = np.einsum("std,td->st", np.abs(H), np.abs(dr))
    units = {}
    for j in range(S):
        units[("ss", j)] = ss[j] + 4 * d * rho[j] ** 2
        units[("g", j)] = G[j]
        units[("z", j)] = P[j] / rho[j] + np.abs(z[j]) + np.abs(z[j] - z.max(axis=0)) + 1
        units[("a", j)] = 2 * a[j]
        units[("dz", j)] = 2 * np.abs(dz[j])
        units[("alpha", j)] = np.abs(alpha[j])
        units[("beta", j)] = 3 * np.abs(beta[j])
    units[("gbar", 0)] = (a * np.abs(g)).sum(axis=0)
    return units, dict(g=g, rho=rho, z=z, a=a, alpha=alpha, beta=beta)


@pytest.mark.parametrize("S,eps,qscale", [(1, 1e-5, 2.0), (2, 1e-5, 1.0), (4, 0.3, 3.0), (6, 1e-5, 0.0),
                                          (9, 1e-5, 4.0)])
def test_backward_scale_sensitivities_match_differences(S, eps, qscale):
    from oracle.attnres_oracle import _backward_core
    H, w, dr = _bwd_case(S, 4, 11, eps, qscale, seed=40 + S)
    units, _ = _model_units(H, w, dr, eps)
    sites = O.backward_rounding_sites(H, w, dr, eps)
    assert {(site, j) for site, j, _ in sites} == set(units)
    for site, j, unit in sites:
        np.testing.assert_allclose(unit, units[(site, j)], rtol=1e-14, atol=0)
    # every site's effect on (a, alpha, beta) by central differences of the
    # evaluation, weighted by its unit, summed in absolute value
    base = _backward_core(H, w, dr, eps)
    want = {k: np.zeros((S, 4)) for k in ("a", "alpha", "beta")}
    for (site, j), unit in units.items():
        x = base[site][j]
        step = 1e-6 * (np.abs(x) + 1e-3 * (1 + np.abs(x).max()))
        bump = np.zeros((1 if site == "gbar" else S, 4))
        bump[j] = step
        up = _backward_core(H, w, dr, eps, bump={site: bump})
        dn = _backward_core(H, w, dr, eps, bump={site: -bump})
        for k in want:
            want[k] += np.abs((up[k] - dn[k]) / (2 * step)) * unit
    got = dict(zip(("a", "alpha", "beta"), O.backward_scalar_sensitivities(H, w, dr, eps)))
    for k in want:
        np.testing.assert_allclose(got[k], want[k], rtol=2e-6, atol=1e-9 * (want[k].max() + 1e-300))
    # the scales are those sensitivities plus one unit per final product and sum
    c = _backward_core(H, w, dr, eps)
    Ak, Bk, Ck = (got[k] + 2 * np.abs(c[k]) for k in ("a", "alpha", "beta"))
    dHs, dws = O.depth_attention_backward_scales(H, w, dr, eps)
    np.testing.assert_allclose(dHs, Ak[:, :, None] * np.abs(dr) + Bk[:, :, None] * np.abs(w) +
                               Ck[:, :, None] * np.abs(H), rtol=1e-14)
    np.testing.assert_allclose(dws, np.einsum("st,std->d", Bk, np.abs(H)), rtol=1e-14)


def test_backward_scale_closed_form_one_source():
    # S = 1: a = 1 and alpha = beta = 0 exactly; only the rounding of the
    # softmax normalisation (a unit of 2) and of gbar = a g (a unit of |g|)
    # reach dz = a (g - gbar), which moves alpha by 1/rho and beta by
    # z / (d rho^2) per unit of dz:
    #   sens_a = 2, sens_alpha = 3|g|/rho, sens_beta = 3|g||z|/(d rho^2)
    rng = np.random.default_rng(8)
    T, d = 5, 24
    H = rng.standard_normal((1, T, d)) * 1.7
    w = rng.standard_normal(d) / 3
    dr = rng.standard_normal((T, d))
    rho = np.sqrt((H[0] ** 2).mean(axis=1) + O.EPS)
    z = H[0] @ w / rho
    g = (H[0] * dr).sum(axis=1)
    sa, sal, sbe = O.backward_scalar_sensitivities(H, w, dr)
    np.testing.assert_allclose(sa[0], 2.0, rtol=1e-14)
    np.testing.assert_allclose(sal[0], 3 * np.abs(g) / rho, rtol=1e-12)
    np.testing.assert_allclose(sbe[0], 3 * np.abs(g * z) / (d * rho ** 2), rtol=1e-12)
    dHs, dws = O.depth_attention_backward_scales(H, w, dr)
    np.testing.assert_allclose(dHs[0], 4 * np.abs(dr) + (3 * np.abs(g) / rho)[:, None] * np.abs(w)
                               + (3 * np.abs(g * z) / (d * rho ** 2))[:, None] * np.abs(H[0]), rtol=1e-12)
    np.testing.assert_allclose(dws, ((3 * np.abs(g) / rho)[:, None] * np.abs(H[0])).sum(axis=0), rtol=1e-12)


def _backward_fp32(H, w, dr, eps):
    """The backward evaluated in float32 (numpy casts only; sums by numpy's
    pairwise float32 summation), as a kernel would."""
    f = np.float32
    h, wq, g_ = H.astype(f), w.astype(f), dr.astype(f)
    S, T, d = H.shape
    rho = np.sqrt(np.sum(h * h, axis=2, dtype=f) / f(d) + f(eps)).astype(f)
    z = (np.sum(h * wq, axis=2, dtype=f) / rho).astype(f)
    e = np.exp(z - z.max(axis=0)).astype(f)
    a = (e / np.sum(e, axis=0, dtype=f)).astype(f)
    g = np.sum(h * g_[None], axis=2, dtype=f)
    gbar = np.sum(a * g, axis=0, dtype=f)
    alpha = (a * (g - gbar) / rho).astype(f)
    beta = (alpha * z / (f(d) * rho)).astype(f)
    dH = a[:, :, None] * g_[None] + alpha[:, :, None] * wq - beta[:, :, None] * h
    dw = np.sum(np.sum(alpha[:, :, None] * h, axis=0, dtype=f), axis=0, dtype=f)
    return dH.astype(np.float64), dw.astype(np.float64)


@pytest.mark.parametrize("d", [64, 1024, 7168])
@pytest.mark.parametrize("S,qscale", [(2, 1.0), (5, 4.0), (9, 1.0), (9, 4.0)])
def test_backward_scale_bounds_a_float32_evaluation(S, d, qscale):
    # an fp32 evaluation errs by at most a few units of u times the scale
    # everywhere (the GPU bars allow 1e-5, about 168 units), and by at least
    # a sixteenth of one unit somewhere in the source gradients (the scale is
    # not inflated); grad_w's scale counts its sum over tokens as if all
    # errors had one sign, so it stays above the error by more
    H, w, dr = _bwd_case(S, 32, d, 1e-5, qscale, seed=S * d)
    H = H.astype(np.float32).astype(np.float64)
    w = w.astype(np.float32).astype(np.float64)
    dr = dr.astype(np.float32).astype(np.float64)
    dH, dw = O.depth_attention_backward(H, w, dr)
    dHs, dws = O.depth_attention_backward_scales(H, w, dr)
    eH, ew = _backward_fp32(H, w, dr, 1e-5)
    rH = np.abs(eH - dH) / (U32 * dHs)
    rw = np.abs(ew - dw) / (U32 * dws)
    assert rH.max() <= 4 and rw.max() <= 4, (rH.max(), rw.max())
    assert rH.max() >= 1 / 16, rH.max()
    assert rw.max() >= 1 / 512, rw.max()


_BACKWARD_SLIPS = [
    ("alpha = dz / rho + ", "alpha = dz + "),                            # missing 1/rho on the logit path
    ("beta = alpha * z / (d * rho) + ", "beta = alpha * z / d + "),      # d rho / d h without 1/rho
    ("- beta[:, :, None] * H", "+ 0 * H"),                               # the rms term dropped
    ("dz = a * (g - gbar) + ", "dz = a * g + "),                         # softmax Jacobian without gbar
    ("a[:, :, None] * dr[None] + alpha", "dr[None] + alpha"),           # value path without a
    ("- beta[:, :, None] * H", "+ beta[:, :, None] * H"),                # wrong sign of the rms term
    ("rho = np.sqrt(ss / d + eps)", "rho = np.sqrt(ss / d)"),            # eps dropped
]


@pytest.mark.parametrize("old,new", _BACKWARD_SLIPS)
def test_backward_bar_rejects_planted_mistakes(old, new):
    # each slip planted in a copy of the oracle's backward moves some
    # gradient entry by more than 100 times the 1e-5 bar of the GPU tests
    import types
    import oracle.attnres_oracle as OA
    src = open(OA.__file__).read()
    assert src.count(old) == 1
    import sys
    mod = types.ModuleType("oracle_with_slip")
    sys.modules[mod.__name__] = mod          # its dataclasses look their module up
    try:
        exec(compile(src.replace(old, new), "oracle_with_slip", "exec"), mod.__dict__)
    finally:
        del sys.modules[mod.__name__]
    rng = np.random.default_rng(17)
    S, T, d = 5, 6, 96
    H = rng.standard_normal((S, T, d)) * np.array([1.0, 0.5, 2.0, 0.003, 1.3])[:, None, None]
    w = rng.standard_normal(d) / math.sqrt(d) * 2
    dr = rng.standard_normal((T, d))
    dH, dw = O.depth_attention_backward(H, w, dr)
    dHs, dws = O.depth_attention_backward_scales(H, w, dr)
    bH, bw = mod.depth_attention_backward(H, w, dr)
    worst = max((np.abs(bH - dH) / (1e-5 * dHs)).max(), (np.abs(bw - dw) / (1e-5 * dws)).max())
    assert worst > 100, worst


# --------------------------------------------------- two-phase merge pin ----

@pytest.mark.parametrize("split", [1, 3, 8])
def test_merge_of_partial_softmaxes_equals_the_union(split):
    # aggregating cached sources first and merging the partial sum in later
    # (the two-phase schedule) must equal one softmax over all sources
    rng = np.random.default_rng(split)
    S, T, d = 9, 5, 32
    H = rng.standard_normal((S, T, d)) * rng.uniform(0.3, 3, size=(S, 1, 1))
    w = rng.standard_normal(d) / math.sqrt(d) * 2
    r_all, a_all = O.depth_attention(H, w)
    r1, a1, l1 = O.depth_attention_lse(H[:split], w)
    r2, a2, l2 = O.depth_attention_lse(H[split:], w)
    r, c1, c2 = O.merge_partial_softmax(r1, l1, r2, l2)
    np.testing.assert_allclose(r, r_all, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(np.concatenate([a1 * c1[:, None], a2 * c2[:, None]], axis=1), a_all,
                               rtol=1e-12, atol=1e-15)
    # lse of a single source is its logit
    _, _, l0 = O.depth_attention_lse(H[:1], w)
    z0 = (O.rmsnorm(H[0]) @ w)
    np.testing.assert_allclose(l0, z0, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------- stack backward -----

def _tiny_grad_stack(L, B, T=2, d=6, seed=0):
    rng = np.random.default_rng(100 + 10 * L + B + seed)
    h0 = rng.standard_normal((T, d))
    W = rng.standard_normal((L + 1, d)) / math.sqrt(d) * 2
    G = rng.standard_normal((L, d))
    Sc = rng.uniform(0.05, 0.2, size=(L, d)) * 5     # larger bodies: every layer matters
    dr = rng.standard_normal((T, d))
    return h0, W, G, Sc, dr


def _stack_loss(h0, W, G, Sc, L, B, dr, full=False):
    fn = lambda l, x: O.synthetic_layer(x, G[l - 1], Sc[l - 1])
    tr = O.full_stack_forward(h0, W, fn, L) if full else O.block_stack_forward(h0, W, fn, L, B)
    return float((tr.r[L] * dr).sum())


@pytest.mark.parametrize("L,B", [(1, 1), (4, 2), (6, 3), (7, 12), (5, 4), (9, 3)])
def test_stack_backward_matches_central_differences(L, B):
    # every entry of dh0 and dW against central differences of the stack
    # forward (a separate code path: explicit value lists and range sums)
    h0, W, G, Sc, dr = _tiny_grad_stack(L, B)
    dh0, dW = O.block_stack_backward(h0, W, G, Sc, L, B, dr)
    step = 1e-6
    for (arr, grad) in ((h0, dh0), (W, dW)):
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += step
            m[idx] -= step
            args_p = (p, W) if arr is h0 else (h0, p)
            args_m = (m, W) if arr is h0 else (h0, m)
            fd = (_stack_loss(*args_p, G, Sc, L, B, dr) - _stack_loss(*args_m, G, Sc, L, B, dr)) / (2 * step)
            assert abs(fd - grad[idx]) <= 1e-7 * (1 + abs(fd)), (idx, fd, grad[idx])


def test_stack_backward_block_size_one_is_full_attnres():
    # block size 1 makes every layer output its own block: the gradients must
    # be those of Full AttnRes, checked by differences of the Full forward
    L = 5
    h0, W, G, Sc, dr = _tiny_grad_stack(L, 1, seed=3)
    dh0, dW = O.block_stack_backward(h0, W, G, Sc, L, 1, dr)
    step = 1e-6
    for idx in [(0, 0), (1, 3), (0, 5)]:
        p, m = h0.copy(), h0.copy()
        p[idx] += step
        m[idx] -= step
        fd = (_stack_loss(p, W, G, Sc, L, 1, dr, full=True) - _stack_loss(m, W, G, Sc, L, 1, dr, full=True)) / (2 * step)
        assert abs(fd - dh0[idx]) <= 1e-7 * (1 + abs(fd))
    for idx in [(0, 1), (3, 2), (5, 4)]:
        p, m = W.copy(), W.copy()
        p[idx] += step
        m[idx] -= step
        fd = (_stack_loss(h0, p, G, Sc, L, 1, dr, full=True) - _stack_loss(h0, m, G, Sc, L, 1, dr, full=True)) / (2 * step)
        assert abs(fd - dW[idx]) <= 1e-7 * (1 + abs(fd))


def test_synthetic_layer_backward_closed_form():
    # d/dx tanh(x g) s at x = 0 is g s; far from zero it vanishes
    g = np.array([0.5, -2.0, 3.0])
    s = np.array([0.1, 0.2, 0.15])
    one = np.ones(3)
    np.testing.assert_allclose(O.synthetic_layer_backward(np.zeros(3), g, s, one), g * s, rtol=0, atol=0)
    assert np.all(np.abs(O.synthetic_layer_backward(np.full(3, 40.0), g, s, one)) < 1e-20)


def test_cpu_rate_process_runs_the_oracle_on_its_slice(tmp_path):
    # the bench's all-cores CPU baseline starts this module once per core;
    # its widening of bf16 bit patterns must be exact and it must report
    # whole chunks of its own tokens
    import json
    import subprocess
    import sys
    import time
    rng = np.random.default_rng(5)
    S, T, d = 3, 40, 16
    x = rng.standard_normal((S, T, d)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16 patterns
    w = (rng.standard_normal(d) / 4).astype(np.float32)
    np.save(tmp_path / "bits.npy", bits)
    np.save(tmp_path / "w.npy", w)
    from oracle.cpu_rate import run
    h = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(h, (x.view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64))
    res = run(str(tmp_path / "bits.npy"), str(tmp_path / "w.npy"), 8, 24, 0.0, 0.05, 8)
    assert res["tokens"] > 0 and res["tokens"] % 8 == 0 and res["end"] >= res["start"]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-m", "oracle.cpu_rate", str(tmp_path / "bits.npy"),
                          str(tmp_path / "w.npy"), "0", "16", repr(time.time()), "0.05", "8"],
                         cwd=root, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert json.loads(out.stdout.strip().splitlines()[-1])["tokens"] > 0
