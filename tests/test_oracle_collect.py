"""Pins of the oracle collect step and of end-to-end oracle invariants.

* The worked example printed on the news repost (refund question): from the
  printed log-probabilities the printed p and residual follow to two decimals.
* Invariants on every question: sum of p is 1; sum of exp(lp) is 1 - residual.
* The floor equals scoring the same question on an empty content, bitwise.
* The results do not depend on the order inputs are submitted in, bitwise.
"""
import json
import os

import numpy as np
import pytest

from oracle import collect as oc
from oracle import plan as op
from oracle import score as osc
from synth import values as sv
from synth import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_refund.json")


def test_worked_example_refund():
    ex = json.load(open(GOLDEN))
    p, residual = oc.option_stats(ex["logprob"])
    tol = 0.5 * 10 ** -ex["printed_decimals"]
    np.testing.assert_allclose(p, ex["p"], atol=tol)
    assert abs(residual - ex["residual"]) <= tol
    # the closed form, with more digits: exp(-0.90) = 0.40657, exp(-1.86) = 0.15567
    np.testing.assert_allclose(p, [0.40657 / 0.56224, 0.15567 / 0.56224], atol=1e-4)
    assert abs(residual - (1 - 0.40657 - 0.15567)) < 1e-4


def test_option_stats_plain_cases():
    p, r = oc.option_stats([np.log(0.5), np.log(0.25)])
    np.testing.assert_allclose(p, [2 / 3, 1 / 3], atol=1e-15)
    assert abs(r - 0.25) < 1e-15
    p, r = oc.option_stats([0.0])
    assert p[0] == 1.0 and r == 0.0


def _oracle_results(inputs, shape, **opts):
    P = op.plan(inputs, vocab=shape.vocab, **opts)
    w = sv.lm_head(shape.vocab, shape.d_model).float().numpy()
    lps = []
    for lay in P.passes:
        keys = sv.path_keys(lay.tok, lay.parent, lay.T)
        rows = lay.slot_row.tolist()
        h = sv.hidden(keys, lay.T_pad, shape.d_model, rows=rows).float().numpy()[rows]
        _, lp = osc.score_rows(h, lay.gather_m, lay.gather_tok, w=w)
        lps.append(lp)
    return P, oc.collect(P, lps)


def test_invariants_on_tiny_and_trie_workloads():
    for inputs in (wl.tiny(), wl.stress(n_questions=12, content_tokens=50, vocab=1024)):
        _, res = _oracle_results(inputs, wl.TINY)
        for per_q in res:
            for r in per_q:
                assert abs(r["p"].sum() - 1) < 1e-14
                assert abs(np.exp(r["lp"]).sum() - (1 - r["residual"])) < 1e-14
                assert abs(r["floor_p"].sum() - 1) < 1e-14
                assert np.all(r["lp"] < 0)


def test_floor_equals_empty_content_input():
    inputs = wl.tiny()
    q = inputs[0][1][2]
    _, res = _oracle_results(inputs + [([], [q])], wl.TINY)
    user = res[0][2]
    empty = res[2][0]
    np.testing.assert_array_equal(user["floor_lp"], empty["lp"])
    np.testing.assert_array_equal(user["floor_p"], empty["p"])
    assert user["floor_residual"] == empty["residual"]


def test_results_do_not_depend_on_submission_order():
    inputs = wl.tiny()
    _, a = _oracle_results(inputs, wl.TINY)
    _, b = _oracle_results(inputs[::-1], wl.TINY)
    for i in range(2):
        for j in range(4):
            for key in ("lp", "p", "floor_lp", "floor_p"):
                np.testing.assert_array_equal(a[i][j][key], b[1 - i][j][key])


def test_multi_token_option_sums_its_tokens():
    inputs = [([1, 2, 3], [([4, 5], [[6, 7], [6, 8], [9]])])]
    P, res = _oracle_results(inputs, wl.TINY, floors=False)
    lay = P.passes[0]
    rec = lay.questions[0]
    keys = sv.path_keys(lay.tok, lay.parent, lay.T)
    rows = lay.slot_row.tolist()
    h = sv.hidden(keys, lay.T_pad, 256, rows=rows).float().numpy()[rows]
    w = sv.lm_head(1024, 256).float().numpy()
    z = h.astype(np.float64) @ w.astype(np.float64).T
    lsm = z - osc.logsumexp(z)[:, None]
    # option [6, 7]: token 6 at the slot (m 0), token 7 at the trie row of (6,) (m 1)
    assert abs(res[0][0]["lp"][0] - (lsm[0, 6] + lsm[1, 7])) < 1e-12
    assert abs(res[0][0]["lp"][2] - lsm[0, 9]) < 1e-12
    assert len(rec.option_gather[0]) == 2
    assert np.isnan(res[0][0]["floor_residual"])
