"""Pins of the layer oracle (rotary positions at tree depth, packed layer) against
mathematics and against unpacked sequences."""
import math

import numpy as np

from oracle import layer as ol
from oracle import plan as op
from synth import workloads as wl


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(0).normal(size=(5, 3, 8))
    assert np.array_equal(ol.rope(x, np.zeros(5), 10000.0), x)


def test_rope_two_dims_is_a_plane_rotation():
    """d = 2: the only frequency is 1, so row p turns by p radians."""
    x = np.random.default_rng(1).normal(size=(6, 1, 2))
    pos = np.arange(6) * 0.7
    got = ol.rope(x, pos, 10000.0)
    for t, p in enumerate(pos):
        r = np.array([[math.cos(p), -math.sin(p)], [math.sin(p), math.cos(p)]])
        assert np.allclose(got[t, 0], r @ x[t, 0], atol=1e-14)


def test_rope_frequencies_by_hand():
    """RoFormer's schedule theta^(-2i/d): with d = 8 and theta = 10^4 the four pairs turn at
    exactly 1, 1/10, 1/100 and 1/1000 radians per position, so a unit vector in pair i
    (components i and i + d/2) at position 10^i turns by one radian, towards the second half."""
    for i in range(4):
        x = np.zeros((1, 1, 8))
        x[0, 0, i] = 1.0
        y = ol.rope(x, [10.0 ** i], 10000.0)[0, 0]
        want = np.zeros(8)
        want[i], want[i + 4] = math.cos(1.0), math.sin(1.0)
        assert np.allclose(y, want, atol=1e-12), i


def test_rope_keeps_pair_norms_and_scores_depend_on_offset_only():
    g = np.random.default_rng(2)
    d = 16
    q, k = g.normal(size=(1, 1, d)), g.normal(size=(1, 1, d))
    x = g.normal(size=(4, 2, d))
    y = ol.rope(x, np.array([3.0, 17.0, 400.0, 9000.0]), 500.0)
    h = d // 2
    assert np.allclose(x[..., :h] ** 2 + x[..., h:] ** 2, y[..., :h] ** 2 + y[..., h:] ** 2)

    def score(m, n):
        return float((ol.rope(q, [m], 500.0) * ol.rope(k, [n], 500.0)).sum())

    for m, n, s in ((5, 2, 11), (40, 40, 3), (9, 30, 100)):
        assert math.isclose(score(m, n), score(m + s, n + s), rel_tol=1e-10, abs_tol=1e-12)


def _unpacked_layer(tokens_x, w_qkv, w_o, Hq, Hkv, d, theta):
    """Textbook causal layer on one unpacked sequence, positions 0..L-1 (no packing)."""
    L = tokens_x.shape[0]
    y = tokens_x @ w_qkv.T
    q = y[:, :Hq * d].reshape(L, Hq, d)
    k = y[:, Hq * d:(Hq + Hkv) * d].reshape(L, Hkv, d)
    v = y[:, (Hq + Hkv) * d:].reshape(L, Hkv, d)
    pos = np.arange(L, dtype=np.float64)
    half = d // 2
    inv = theta ** (-2.0 * np.arange(half) / d)

    def turn(x):
        a = pos[:, None] * inv[None, :]
        c, s = np.cos(a)[:, None, :], np.sin(a)[:, None, :]
        return np.concatenate([x[..., :half] * c - x[..., half:] * s, x[..., half:] * c + x[..., :half] * s], -1)

    q, k = turn(q), turn(k)
    o = np.zeros((L, Hq, d))
    for h in range(Hq):
        g = h * Hkv // Hq
        s = q[:, h, :] @ k[:, g, :].T / math.sqrt(d)
        s = np.where(np.tril(np.ones((L, L), dtype=bool)), s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        o[:, h, :] = (p / p.sum(axis=1, keepdims=True)) @ v[:, g, :]
    return o.reshape(L, Hq * d) @ w_o.T


def test_packed_layer_equals_each_unpacked_branch():
    """Every row of a packed pass (content rows, question rows, option-prefix rows)
    gets the layer output of its own unpacked sequence at positions 0..L-1."""
    g = np.random.default_rng(3)
    Hq, Hkv, d, D, theta = 4, 2, 8, 16, 100.0
    inputs = wl.stress(n_questions=3, content_tokens=12, vocab=50) + [([], [([2, 3], [[4], [5, 6]])])]
    lay = op.plan(inputs, token_budget=256, vocab=50).passes[0]
    emb = g.normal(size=(50, D))          # a token's input row is its embedding
    x = emb[lay.tok]
    w_qkv, w_o = g.normal(size=((Hq + 2 * Hkv) * d, D)) / math.sqrt(D), g.normal(size=(D, Hq * d)) / math.sqrt(Hq * d)
    rows = list(range(lay.T))
    got = ol.packed_layer_rows(lay, x, w_qkv, w_o, Hq, Hkv, d, theta, rows)
    for r in rows:
        path = lay.visible(r)                      # the row's unpacked sequence, in order
        ref = _unpacked_layer(emb[lay.tok[path]], w_qkv, w_o, Hq, Hkv, d, theta)[-1]
        assert np.allclose(got[r], ref, atol=1e-10), r


def test_static_quantisation_matches_torch_recipe():
    """e4m3 codes with a static scale against torch's float8_e4m3fn cast of the fp32
    quotient (clamped to +-448 first: torch's cast does not saturate)."""
    import torch
    g = np.random.default_rng(5)
    x = (g.standard_normal((40, 96)) * 3).astype(np.float32)
    x[0, :4] = [0.0, -0.0, 1e-9, 5000.0]
    s = np.float32(0.0123)
    codes = ol.quantize_static(x, s)
    q = torch.from_numpy(x) / torch.tensor(s)
    want = torch.clamp(q, -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, want)


def test_fp8_linear_against_torch_decoded_values():
    import torch
    g = np.random.default_rng(6)
    xc = g.integers(0, 256, size=(7, 64)).astype(np.uint8)
    wc = g.integers(0, 256, size=(9, 64)).astype(np.uint8)
    xc[(xc & 0x7F) == 0x7F] = 0   # no NaN codes
    wc[(wc & 0x7F) == 0x7F] = 0
    ws = g.random(9).astype(np.float32) + 0.5
    xs = np.float32(0.37)
    y = ol.linear_fp8(xc, xs, wc, ws)
    xd = torch.from_numpy(xc).view(torch.float8_e4m3fn).double() * float(xs)
    wd = torch.from_numpy(wc).view(torch.float8_e4m3fn).double() * torch.from_numpy(ws).double()[:, None]
    np.testing.assert_allclose(y, (xd @ wd.T).numpy(), rtol=1e-13, atol=1e-13)


def test_qkv_rope_is_projection_then_rotation():
    g = np.random.default_rng(8)
    T, D, Hq, Hkv, d = 5, 32, 2, 1, 16
    x = g.standard_normal((T, D))
    w = g.standard_normal(((Hq + 2 * Hkv) * d, D))
    pos = np.array([0, 3, 1, 7, 2])
    q, k, v = ol.qkv_rope(x, w, pos, Hq, Hkv, d, 10000.0)
    y = x @ w.T
    # position 0 leaves the row unturned; v is never turned
    np.testing.assert_allclose(q[0].reshape(-1), y[0, :Hq * d], rtol=0, atol=1e-12)
    np.testing.assert_allclose(v.reshape(T, -1), y[:, (Hq + Hkv) * d:], rtol=0, atol=1e-12)
    # a turn keeps each pair's norm
    kk = y[:, Hq * d:(Hq + Hkv) * d].reshape(T, Hkv, d)
    np.testing.assert_allclose(np.hypot(k[..., :d // 2], k[..., d // 2:]),
                               np.hypot(kk[..., :d // 2], kk[..., d // 2:]), rtol=1e-12)


def test_qkv_rope_turns_q_and_k_by_their_own_positions():
    """Rows with the same input at positions (5, 2) and (15, 12): each q . k score depends on
    the offset only, which holds only if both q and k are turned by their rows' positions."""
    g = np.random.default_rng(9)
    D, Hq, Hkv, d = 32, 2, 1, 16
    x = np.repeat(g.standard_normal((1, D)), 4, axis=0)
    w = g.standard_normal(((Hq + 2 * Hkv) * d, D))
    q, k, _ = ol.qkv_rope(x, w, np.array([5, 2, 15, 12]), Hq, Hkv, d, 10000.0)
    for h in range(Hq):
        assert math.isclose(q[0, h] @ k[1, 0], q[2, h] @ k[3, 0], rel_tol=1e-10)
    assert not math.isclose(q[0, 0] @ k[1, 0], q[0, 0] @ k[3, 0], rel_tol=1e-6)   # the offset does matter
