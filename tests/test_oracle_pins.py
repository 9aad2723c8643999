"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test names what fixes the expected values: a hand-worked fixture, a
closed form, exact rational brute force, an invariant, or a library routine
that a special case reduces to.  Page citations are to "Skipping dead
neurons: a faster Nemotron 3.5 Lightning on Apple silicon" (sevren.ai).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from synth import W4Proj, Expert

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _proj(codes, scale, bias):
    return W4Proj(torch.as_tensor(np.asarray(codes, dtype=np.uint8)),
                  torch.as_tensor(np.asarray(scale, dtype=np.float16)),
                  torch.as_tensor(np.asarray(bias, dtype=np.float16)))


def _pack(q):
    """Pack integer codes [rows][cols] (low nibble = even column); written here
    from the layout statement, independently of the oracle's unpacking."""
    q = np.asarray(q, dtype=np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def _rand_proj(rng, rows, cols):
    q = rng.integers(0, 16, size=(rows, cols))
    s = rng.uniform(0.002, 0.02, size=(rows, cols // 64)).astype(np.float16)
    b = (rng.uniform(-0.2, 0.2, size=(rows, cols // 64))).astype(np.float16)
    return _proj(_pack(q), s, b), q


# ---------------------------------------------------------------- layout ----

def test_dequant_layout_golden():
    """Hand-built bytes -> hand-worked weights (section "The whole decode step":
    one scale per group of 64; packing order as read in the fixture)."""
    g = _read_golden("w4_layout.txt")
    sc = [float(v) for v in g[0][1:]]
    bi = [float(v) for v in g[1][1:]]
    row0 = np.full(64, 0x21, dtype=np.uint8)
    row1 = np.array([((j % 16) << 4) | (15 - j % 16) for j in range(64)], dtype=np.uint8)
    p = _proj(np.stack([row0, row1]), [[sc[0], sc[1]], [sc[2], sc[3]]],
              [[bi[0], bi[1]], [bi[2], bi[3]]])
    w = oracle.dequant(p)
    assert w.shape == (2, 128)
    for r, c, v in g[2:]:
        assert w[int(r), int(c)] == float(v), (r, c)


def test_unpack_codes_roundtrip_bytes():
    b = np.arange(256, dtype=np.uint8).reshape(2, 128)
    q = oracle.unpack_codes(b)
    assert (q[:, 0::2] == (b & 15)).all() and (q[:, 1::2] == (b >> 4)).all()
    assert q.max() == 15 and q.min() == 0


# ------------------------------------------------------------ ReLU^2 -------

def test_relu2_twelve_neurons_golden():
    """The hand-worked 12-neuron example (section "Transposing to skip the zeros";
    the page's own numbers were lost, these are worked by hand in the fixture)."""
    g = {r[0]: r[1:] for r in _read_golden("relu2_12.txt")}
    z = np.array([float(v) for v in g["z"]])
    h = oracle.relu2(z)
    assert h.tolist() == [float(v) for v in g["h"]]
    assert oracle.live_set(h).tolist() == [int(v) for v in g["live"]]
    # down projection of the padded example, hand sums in the fixture
    hz = np.concatenate([z, -np.ones(52)])
    hp = oracle.relu2(hz)
    q = np.array([[(n + 3 * o) % 16 for n in range(64)] for o in range(4)])
    down = _proj(_pack(q), np.ones((4, 1)), -8 * np.ones((4, 1)))
    y = oracle.down_dense(hp, down)
    assert y.tolist() == [float(v) for v in g["y"]]
    assert oracle.down_sparse_sequential(hp, down).tolist() == [float(v) for v in g["y"]]


def test_relu2_edge_values():
    z = np.array([-0.0, 0.0, -np.inf, np.inf, 1e-200, -1e-200, 2.0 ** -600])
    h = oracle.relu2(z)
    assert h[0] == 0 and h[1] == 0 and h[2] == 0 and h[3] == np.inf
    assert h[4] == 0.0  # squares underflow: counts as dead
    assert oracle.live_set(h).tolist() == [3]


# ------------------------------------------------------------ down ---------

def test_down_closed_form_constant_codes():
    """All codes of group g equal c_g  =>  y_o = sum_g (s_og c_g + b_og) * sum_{n in g} h_n."""
    rng = np.random.default_rng(1)
    rows, N = 16, 256
    c = np.array([3, 0, 15, 9])
    q = np.repeat(c[None, :], rows, 0).repeat(64, 1)
    s = rng.uniform(0.002, 0.02, (rows, 4)).astype(np.float16)
    b = rng.uniform(-0.1, 0.1, (rows, 4)).astype(np.float16)
    h = oracle.relu2(rng.normal(-1.0, 1.0, N))
    y = oracle.down_dense(h, _proj(_pack(q), s, b))
    hg = h.reshape(4, 64).sum(1)
    exp = ((s.astype(np.float64) * c + b.astype(np.float64)) * hg).sum(1)
    np.testing.assert_allclose(y, exp, rtol=1e-13, atol=1e-15)


def test_down_one_hot_reads_column():
    """h = v e_n  =>  y_o = v * (s[o, n//64] * q[o, n] + b[o, n//64]); q read from the byte."""
    rng = np.random.default_rng(2)
    rows, N = 8, 192
    p, q = _rand_proj(rng, rows, N)
    bytes_ = p.codes.numpy()
    for n in (0, 1, 63, 64, 65, 130, 191):
        h = np.zeros(N)
        h[n] = 2.5
        y = oracle.down_dense(h, p)
        for o in range(rows):
            byte = int(bytes_[o, n // 2])
            code = (byte >> 4) if n % 2 else (byte & 15)
            w = float(p.scale[o, n // 64]) * code + float(p.bias[o, n // 64])
            assert y[o] == 2.5 * w


def test_down_exact_rational_brute_force():
    """Tiny shapes, every live mask over 12 chosen neurons: fp64 result vs the
    exact rational sum (Fractions) of the definition."""
    rng = np.random.default_rng(3)
    for N in (64, 128):
        rows = 64
        p, q = _rand_proj(rng, rows, N)
        sF = [[Fraction(float(v)) for v in r] for r in p.scale.numpy()]
        bF = [[Fraction(float(v)) for v in r] for r in p.bias.numpy()]
        chosen = rng.choice(N, 12, replace=False)
        hv = rng.uniform(0.01, 3.0, 12)
        W = oracle.dequant(p)
        masks = list(range(4096))
        for m in masks:
            h = np.zeros(N)
            for i in range(12):
                if (m >> i) & 1:
                    h[chosen[i]] = hv[i]
            y = oracle.down_dense(h, p)
            ys = oracle.down_sparse_sequential(h, p)
            assert (ys == oracle.down_dense_sequential(h, p)).all()
            if m % 257 == 0:  # exact check on a sample of masks (Fractions are slow)
                for o in range(0, rows, 7):
                    ex = sum((sF[o][n // 64] * int(q[o, n]) + bF[o][n // 64]) * Fraction(h[n])
                             for n in range(N) if h[n] != 0)
                    assert abs(Fraction(y[o]) - ex) <= Fraction(1, 10**12) * (1 + abs(ex))
            # the dense product with W gives the same up to fp64 rounding
            np.testing.assert_allclose(y, W @ h, rtol=1e-12, atol=1e-12)


def test_sparse_equals_dense_bit_exact_full_width():
    """Sparse form over live rows == dense form over all rows, bit for bit in fp64
    ("Our way reads only the rows that fired": same answer)."""
    rng = np.random.default_rng(4)
    p, _ = _rand_proj(rng, 2688, 256)
    h = oracle.relu2(rng.normal(-1.28, 1.0, 256))
    a = oracle.down_sparse_sequential(h, p)
    b = oracle.down_dense_sequential(h, p)
    assert np.array_equal(a, b)


def test_down_linearity():
    rng = np.random.default_rng(5)
    p, _ = _rand_proj(rng, 64, 128)
    h1 = oracle.relu2(rng.normal(-1, 1, 128))
    h2 = oracle.relu2(rng.normal(-1, 1, 128))
    np.testing.assert_allclose(oracle.down_dense(h1 + h2, p),
                               oracle.down_dense(h1, p) + oracle.down_dense(h2, p), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ up -----------

def test_up_closed_form_and_one_hot():
    rng = np.random.default_rng(6)
    N, H = 8, 192
    c = np.array([1, 14, 7])
    q = np.repeat(c[None, :], N, 0).repeat(64, 1)
    s = rng.uniform(0.002, 0.02, (N, 3)).astype(np.float16)
    b = rng.uniform(-0.1, 0.1, (N, 3)).astype(np.float16)
    up = _proj(_pack(q), s, b)
    off = rng.normal(0, 1, N).astype(np.float32)
    x = rng.normal(0, 1, H).astype(np.float32)
    z = oracle.up_preact(x, up, off)
    X = x.astype(np.float64).reshape(3, 64).sum(1)
    exp = ((s.astype(np.float64) * c + b.astype(np.float64)) * X).sum(1) + off
    np.testing.assert_allclose(z, exp, rtol=1e-12, atol=1e-12)
    # one-hot x picks a single weight; the offset is added once
    p, qq = _rand_proj(rng, N, H)
    for k in (0, 63, 64, 191):
        xe = np.zeros(H)
        xe[k] = -1.5
        z = oracle.up_preact(xe, p, off)
        w = p.scale.numpy()[:, k // 64].astype(np.float64) * qq[:, k] + p.bias.numpy()[:, k // 64]
        assert np.array_equal(z, -1.5 * w + off.astype(np.float64))


def test_up_batched_equals_single():
    rng = np.random.default_rng(7)
    p, _ = _rand_proj(rng, 16, 128)
    X = rng.normal(0, 1, (5, 128))
    Z = oracle.up_preact(X, p)
    for t in range(5):
        np.testing.assert_allclose(Z[t], oracle.up_preact(X[t], p), rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------ router -------

def test_router_ties_and_order():
    """Top-6 of 128 ("Inside a MoE layer"); ties to the lower index (reading)."""
    l = np.full(128, -5.0)
    l[[1, 2, 4, 5, 6, 0, 77]] = [3, 3, 2, 2, 2, 1, 1]
    idx, w = oracle.router_topk(l, 6)
    assert idx.tolist() == [1, 2, 4, 5, 6, 0]
    # softmax over the 6 chosen only: independent of the other 122 logits
    l2 = l.copy()
    l2[100:] = 0.5
    idx2, w2 = oracle.router_topk(l2, 6)
    assert idx2.tolist() == idx.tolist() and np.array_equal(w, w2)
    e = np.exp([0, 0, -1, -1, -1, -2])
    np.testing.assert_allclose(w, e / e.sum(), rtol=1e-15)


def test_router_softmax_closed_forms():
    l = np.zeros(128)
    l[10:16] = 7.25
    idx, w = oracle.router_topk(l, 6)
    assert idx.tolist() == list(range(10, 16))
    np.testing.assert_allclose(w, np.full(6, 1 / 6), rtol=1e-15)
    l = np.zeros(128)
    l[3], l[9] = math.log(2.0) + 4.0, 4.0
    l[20:24] = -50.0 + np.arange(4)
    l[:3] = -100
    idx, w = oracle.router_topk(l, 2)
    assert idx.tolist() == [3, 9]
    np.testing.assert_allclose(w, [2 / 3, 1 / 3], rtol=1e-14)
    rng = np.random.default_rng(8)
    idx, w = oracle.router_topk(rng.normal(size=(50, 128)), 6)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-15)
    assert (np.diff(w, axis=1) <= 0).all()


def test_router_projection_hand_values_and_selectors():
    """The router projection (reading of "Inside a MoE layer": one logit per
    expert, a linear map of x): a hand-worked 3 x 4 case, selector rows that
    must return single entries of x (a transposed W or a wrong axis fails),
    an all-ones row that must return the exact sum, and linearity."""
    x = np.array([1.0, 2.0, -3.0, 0.5])
    W = np.array([[1.0, 0.0, 0.0, 0.0], [0.5, 0.5, 0.5, 0.5], [-1.0, 2.0, 0.0, 4.0]])
    assert oracle.router_logits(x, W).tolist() == [1.0, 0.25, 5.0]
    rng = np.random.default_rng(21)
    H, E = 64, 8
    xs = rng.integers(-64, 64, size=(3, H)) / 8.0           # dyadic: every sum below is exact in fp64
    sel = np.zeros((E, H))
    cols = [5, 0, 63, 17, 17, 2, 40, 9]
    sel[np.arange(E), cols] = 1.0
    L = oracle.router_logits(xs, sel)
    assert L.shape == (3, E) and np.array_equal(L, xs[:, cols])
    ones = np.ones((1, H))
    assert oracle.router_logits(xs[0], ones)[0] == math.fsum(xs[0])
    Wr = rng.integers(-8, 8, size=(E, H)) / 4.0
    np.testing.assert_array_equal(oracle.router_logits(xs[0] + xs[1], Wr),
                                  oracle.router_logits(xs[0], Wr) + oracle.router_logits(xs[1], Wr))


# ------------------------------------------------- row-scale requant ------

def _ckpt(H, N, codes_fn, scale=1.0, bias=-8.0):
    """A checkpoint-layout projection [H][N] with constant scale and bias."""
    q = np.fromfunction(codes_fn, (H, N), dtype=np.int64).astype(np.uint8) & 15
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    s = np.full((H, N // 64), scale, dtype=np.float16)
    b = np.full((H, N // 64), bias, dtype=np.float16)
    return type("P", (), {"codes": packed, "scale": s, "bias": b})()


def test_requant_rowscale_hand_group_and_round_trip():
    """Re-quantisation along the neuron axis ("The whole decode step"):
    (a) a hand-worked group: neuron 1's 64 outputs take the values
    1 + 0.5 k (k = 0..15, each four times) -> scale 0.5, bias 1, codes k;
    (b) integer weights whose every (neuron, 64-output) group spans -8..7
    come back exactly (scale 1, bias -8, the checkpoint's own codes);
    (c) a constant group gets scale 0 and codes 0."""
    H, N = 64, 64
    # checkpoint scale 0.5, bias 1 on neuron group 0: w = 0.5 q + 1
    k_of_o = np.arange(64) % 16
    P = _ckpt(H, N, lambda o, n: np.where(n == 1, k_of_o[o], 3), scale=0.5, bias=1.0)
    codes, s, b = oracle.requant_down_rowscale(P)
    assert s.shape == (N, 1) and codes.shape == (N, 32)
    assert float(s[1, 0]) == 0.5 and float(b[1, 0]) == 1.0
    q1 = oracle.unpack_codes(codes)[1]
    assert q1.tolist() == k_of_o.tolist()
    assert float(s[0, 0]) == 0.0 and float(b[0, 0]) == 2.5 and not oracle.unpack_codes(codes)[0].any()  # w = 2.5
    # (b) round trip on groups spanning the full 16-value grid
    H, N = 256, 192
    rng = np.random.default_rng(31)
    Q = rng.integers(0, 16, size=(H, N))
    Q[0::64, :] = 0
    Q[1::64, :] = 15
    P = _ckpt(H, N, lambda o, n: Q[o, n])
    codes, s, b = oracle.requant_down_rowscale(P)
    assert (s == 1.0).all() and (b == -8.0).all()
    np.testing.assert_array_equal(oracle.dequant_rowscale(codes, s, b), oracle.dequant(P))
    np.testing.assert_array_equal(oracle.unpack_codes(codes), Q.T)


def test_requant_rowscale_error_within_one_step():
    """Random checkpoint weights: every re-quantised weight lies within one
    step (its own group's scale) of the original; scales are positive and
    follow the range of their own (neuron, 64-output) group."""
    import synth
    H, N = 256, 128
    down = synth.gen_proj(H, N, (3, "requant-pin"))
    W = oracle.dequant(down)
    codes, s, b = oracle.requant_down_rowscale(down)
    Wr = oracle.dequant_rowscale(codes, s, b)
    step = np.repeat(s.astype(np.float64), 64, axis=-1).T     # [H][N]
    assert (np.abs(Wr - W) <= step * 0.51 + 1e-3 * step + 2.0 ** -20).all()
    rng_ = W.T.reshape(N, H // 64, 64)
    np.testing.assert_allclose(s.astype(np.float64), (rng_.max(2) - rng_.min(2)) / 15, rtol=2e-3)


# ------------------------------------------------------------ layer --------

def _tiny_expert(rng, N, H, zero=False):
    up, _ = _rand_proj(rng, N, H)
    if zero:
        s = rng.uniform(0.002, 0.02, (H, N // 64)).astype(np.float16)
        down = _proj(np.full((H, N // 2), 0x88, np.uint8), s, (-8 * s.astype(np.float32)).astype(np.float16))
    else:
        down, _ = _rand_proj(rng, H, N)
    off = torch.from_numpy(rng.normal(0, 0.05, N).astype(np.float32))
    return Expert(up, down, off)


def test_layer_shared_only_when_routed_are_zero():
    """Routed experts whose down weights dequantise to 0 (code 8, bias -8*scale)
    leave exactly the shared expert's output ("Inside a MoE layer")."""
    rng = np.random.default_rng(9)
    H = 128
    zeros = {e: _tiny_expert(rng, 64, H, zero=True) for e in range(16)}
    shared = _tiny_expert(rng, 128, H)
    x = torch.from_numpy(rng.normal(0, 1, H).astype(np.float32))
    lg = rng.normal(0, 1, 16)
    r = oracle.moe_layer(x, lg, lambda e: zeros[e], shared, k=6)
    assert np.array_equal(r["out"], oracle.expert_forward(x, shared)["y"])


def test_layer_identical_routed_experts_sum_to_one():
    """Six identical routed experts, no shared: out = y_e * sum(w) = y_e."""
    rng = np.random.default_rng(10)
    H = 128
    ex = _tiny_expert(rng, 64, H)
    x = torch.from_numpy(rng.normal(0, 1, H).astype(np.float32))
    r = oracle.moe_layer(x, rng.normal(0, 1, 32), lambda e: ex, None, k=6)
    np.testing.assert_allclose(r["out"], oracle.expert_forward(x, ex)["y"], rtol=1e-13, atol=1e-13)


def test_layer_weighting_matches_hand_combination():
    rng = np.random.default_rng(11)
    H = 128
    exs = {e: _tiny_expert(rng, 64, H) for e in range(8)}
    shared = _tiny_expert(rng, 128, H)
    x = torch.from_numpy(rng.normal(0, 1, H).astype(np.float32))
    lg = np.array([0.1, 2.0, -1.0, 0.5, 1.5, -0.2, 0.7, 0.0])
    r = oracle.moe_layer(x, lg, lambda e: exs[e], shared, k=6)
    order = [1, 4, 6, 3, 0, 7]
    assert r["idx"].tolist() == order
    ex = np.exp(lg[order] - 2.0)
    w = ex / ex.sum()
    y = oracle.expert_forward(x, shared)["y"].copy()
    for j, e in enumerate(order):
        y += w[j] * oracle.expert_forward(x, exs[e])["y"]
    np.testing.assert_allclose(r["out"], y, rtol=1e-13, atol=1e-13)


def test_tokens_equal_per_token_layer():
    """Batch/prefill form == the one-token definition applied to each token."""
    rng = np.random.default_rng(12)
    H = 128
    exs = {e: _tiny_expert(rng, 64, H) for e in range(10)}
    shared = _tiny_expert(rng, 128, H)
    X = rng.normal(0, 1, (7, H))
    L = rng.normal(0, 1, (7, 10))
    r = oracle.moe_tokens(X, L, lambda e: exs[e], shared, k=6)
    for t in range(7):
        one = oracle.moe_layer(X[t], L[t], lambda e: exs[e], shared, k=6)
        np.testing.assert_allclose(r["out"][t], one["out"], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ bf16 ---------

def test_bf16_rne_hand_values():
    v = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -30, -(1 + 2 ** -8),
                  1.5 * 2 ** -133, 2.5 * 2 ** -133, 3.0e38, 3.4e38, 0.0, -0.0, np.inf])
    r = oracle.bf16_rne(v)
    # ties go to the even neighbour; 3.0e38 / 2^127 = 1.7632 -> 226/128; 3.4e38 is past
    # the midpoint between the largest bf16 value (2 - 2^-7) * 2^127 and 2^128 -> inf
    exp = [1.0, 1 + 2 ** -6, 1 + 2 ** -7, -1.0, 2 ** -132, 2 ** -132, 226 / 128 * 2.0 ** 127,
           np.inf, 0.0, -0.0, np.inf]
    assert r.tolist() == exp
    assert np.signbit(r[9])


def test_bf16_rne_matches_library_on_fp32_values():
    """For fp32-representable inputs, direct RNE from fp64 equals torch's fp32->bf16."""
    rng = np.random.default_rng(13)
    v = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-30, 2000),
                        rng.normal(0, 1e30, 2000)]).astype(np.float32)
    # include exact ties
    t = (rng.integers(1, 2 ** 8, 1000) * 2 + 1).astype(np.float64) * 2.0 ** -9
    v = np.concatenate([v, t.astype(np.float32)])
    lib = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(oracle.bf16_rne(v.astype(np.float64)), lib)


# ------------------------------------------------------------ bytes --------

def test_down_required_bytes_closed_form():
    """One live neuron costs a row (hidden/2 B) and its group's scales (hidden*4 B);
    a fully dead group costs nothing (section "The whole decode step")."""
    h = np.zeros(256)
    assert oracle.down_required_bytes(h, 2688) == 0
    h[5] = 1.0
    assert oracle.down_required_bytes(h, 2688) == 1344 + 10752
    h[6] = 2.0
    h[200] = 1.0
    assert oracle.down_required_bytes(h, 2688) == 3 * 1344 + 2 * 10752
