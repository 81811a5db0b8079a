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
