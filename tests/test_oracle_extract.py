"""Pins of the oracle's searched slots ({*}, {n}, {$}): layout, top-k selection, collection.

The layout arrays were worked out by hand from the layout rules (a searched slot
lays out its template only; its last template row is a scoring row; it gets no
floor).  The top-k cases are hand-ordered lists, a brute-force selection on small
random inputs, and logits made exact by a one-hot hidden row.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import collect as oc
from oracle import plan as op
from oracle import score as osc


def test_searched_slot_layout_by_hand():
    req = [([10, 11], [([20, 21], [[30], [31]]), ([40, 41, 42], None, -1), ([50], [[60, 61], [62]])])]
    P = op.plan(req)
    assert len(P.passes) == 1
    L = P.passes[0]
    # user rows 0-8 (content, q0, searched q1, q2 with trie node (60,)), floors of q0 and q2 only
    assert L.T == 13
    assert L.tok[:13].tolist() == [10, 11, 20, 21, 40, 41, 42, 50, 60, 20, 21, 50, 60]
    assert L.parent[:13].tolist() == [-1, 0, 1, 2, 1, 4, 5, 1, 7, -1, 9, -1, 11]
    assert L.pos[:13].tolist() == [0, 1, 2, 3, 2, 3, 4, 2, 3, 0, 1, 0, 1]
    assert L.end[:13].tolist() == [9, 9, 4, 4, 7, 7, 7, 9, 9, 11, 11, 13, 13]
    assert L.anchor[:13].tolist() == [0] * 9 + [9, 9, 11, 11]
    assert L.slot_row.tolist() == [3, 6, 7, 8, 10, 11, 12]
    assert L.gather_m.tolist() == [0, 0, 2, 3, 2, 4, 4, 5, 6, 5]
    assert L.gather_tok.tolist() == [30, 31, 60, 61, 62, 30, 31, 60, 61, 62]
    assert L.x_m.tolist() == [1] and L.x_set.tolist() == [-1]
    assert L.tile_ptr.tolist() == [0, 3]
    assert L.tile_kv.tolist() == [0, 9, 11] and L.tile_len.tolist() == [9, 2, 2]
    assert L.visible(6) == [0, 1, 4, 5, 6]
    assert P.n_options == [[2, 0, 2]] and P.searched == [[False, True, False]]
    assert len(P.floor_home) == 2


def test_searched_slot_validation():
    with pytest.raises(op.PlanError) as e:
        op.plan([([1], [([2], None, -2)])])
    assert e.value.status == "INVALID"
    with pytest.raises(op.PlanError) as e:
        op.plan([([1], [([], None, 0)])])
    assert e.value.status == "INVALID"
    with pytest.raises(op.PlanError) as e:
        op.plan([([1], [([2], None, 0)])], extract_k=0)
    assert e.value.status == "INVALID"
    with pytest.raises(op.PlanError) as e:
        op.plan([([1], [([2], [])])])   # a scored question still needs options
    assert e.value.status == "INVALID"


Z16 = np.array([3, 1, 4, 1, 5, 9, 2, 6, 5, 3, 5, 8, 9, 7, 9, 3], dtype=np.float64)


def test_topk_by_hand():
    lse = float(logsumexp(Z16))
    tok, lp = osc.topk_allowed(Z16, lse, None, 4)
    assert tok.tolist() == [5, 12, 14, 11]          # three 9s by token id, then the 8
    np.testing.assert_allclose(lp, [9 - lse, 9 - lse, 9 - lse, 8 - lse], rtol=0, atol=1e-12)
    allowed = np.zeros(16, bool)
    allowed[[1, 3, 7, 13]] = True
    tok, _ = osc.topk_allowed(Z16, lse, allowed, 3)
    assert tok.tolist() == [13, 7, 1]                # 7, 6, then the lower of the two 1s
    only = np.zeros(16, bool)
    only[2] = True
    tok, lp = osc.topk_allowed(Z16, lse, only, 3)
    assert tok.tolist() == [2, -1, -1]
    assert lp[0] == pytest.approx(4 - lse, abs=1e-12) and np.isneginf(lp[1:]).all()


def _brute_topk(z, allowed, k):
    chosen = []
    for _ in range(k):
        best = None
        for v in range(len(z)):
            if (allowed is not None and not allowed[v]) or v in chosen:
                continue
            if best is None or z[v] > z[best]:   # scanning upwards keeps the lower id on ties
                best = v
        if best is None:
            break
        chosen.append(best)
    return chosen + [-1] * (k - len(chosen))


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force(seed):
    g = np.random.default_rng(seed)
    V = int(g.integers(5, 60))
    z = g.integers(-4, 5, size=V).astype(np.float64)   # many ties
    allowed = g.random(V) < 0.5 if seed % 2 else None
    k = int(g.integers(1, 17))
    lse = float(logsumexp(z))
    tok, lp = osc.topk_allowed(z, lse, allowed, k)
    assert tok.tolist() == _brute_topk(z, allowed, k)
    for t, l in zip(tok, lp):
        assert (t < 0 and l == -np.inf) or l == pytest.approx(z[t] - lse, abs=1e-12)


def test_extract_rows_with_exact_logits():
    # hidden rows e0 and 2 e0: z[v] = W[v, 0] * {1, 2}, exact in fp64
    V, D = 16, 8
    g = np.random.default_rng(1)
    w = np.zeros((V, D))
    w[:, 0] = Z16
    w[:, 1:] = g.standard_normal((V, D - 1))
    h = np.zeros((2, D))
    h[0, 0], h[1, 0] = 1.0, 2.0
    sets = [np.isin(np.arange(V), [1, 3, 7, 13])]
    tok, lp = osc.extract_rows(h, [-1, 0], sets, 4, w=w)
    assert tok[0].tolist() == [5, 12, 14, 11]
    assert tok[1].tolist() == [13, 7, 1, 3]
    lse1 = math.log(sum(math.exp(2 * v) for v in Z16))
    np.testing.assert_allclose(lp[1], [14 - lse1, 12 - lse1, 2 - lse1, 2 - lse1], rtol=0, atol=1e-12)


def test_collect_extract_maps_question_order():
    # two inputs that cannot share a pass; each has a searched slot between scored questions
    req = [([1] * 10, [([2, 3], [[4], [5]]), ([6, 7], None, 0)]),
           ([8] * 10, [([9], None, -1), ([2, 3], [[4], [5]]), ([6], None, 1)])]
    P = op.plan(req, token_budget=16, floors=False)
    assert len(P.passes) == 2
    assert [L.x_set.tolist() for L in P.passes] == [[0], [-1, 1]]
    k = P.extract_k
    tok = [np.array([[100 * p + x] * k for x in range(len(L.x_m))]) for p, L in enumerate(P.passes)]
    lp = [-(t.astype(np.float64)) for t in tok]
    out = oc.collect_extract(P, tok, lp)
    assert [int(t[0]) for t, _ in out] == [0, 100, 101]
    res = oc.collect(P, [np.zeros(len(L.gather_tok)) for L in P.passes])
    assert res[0][1] is None and res[1][0] is None and res[1][2] is None
    assert res[1][1]["p"].sum() == pytest.approx(1.0)
