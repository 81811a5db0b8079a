"""Oracle result collection in fp64 (TEST INFRASTRUCTURE ONLY).

Restates "spinf-serve 0.1.1" (PyPI), "What it does" and the worked example of
the "spinf-serve" news repost (the refund question's response fragment):

* an option's log-probability is the sum of its token log-probabilities
  (a multi-token option reads its later tokens at its trie rows);
* ``p`` is the probability among the question's options:
  ``p_o = exp(lp_o) / sum_j exp(lp_j)``;
* ``residual`` is the probability that went outside the options:
  ``1 - sum_j exp(lp_j)`` (not clamped; it can only go negative when one option
  is a token prefix of another);
* ``floor_*`` are the same quantities for the same question on empty content.

A searched slot's answer (tokens and their log-probabilities, see
:func:`oracle.score.topk_allowed`) is reported as it comes out of its pass.
"""
from __future__ import annotations

import numpy as np


def option_stats(lp):
    """``(p, residual)`` of one question from its option log-probabilities."""
    lp = np.asarray(lp, dtype=np.float64)
    m = lp.max()
    e = np.exp(lp - m)
    p = e / e.sum()
    residual = -np.expm1(m + np.log(e.sum()))
    return p, residual


def collect(plan, token_lp_per_pass):
    """Per user question: option lp, p, residual and their floors.

    ``token_lp_per_pass[p]`` holds the token log-probabilities of pass ``p`` in
    gather order.  Returns a list (per input) of lists (per question) of dicts.
    """
    def question_lp(home):
        p, idx = home
        rec = plan.passes[p].questions[idx]
        tl = np.asarray(token_lp_per_pass[p], dtype=np.float64)
        out = []
        for gs in rec.option_gather:
            acc = 0.0
            for g in gs:                      # token order
                acc += float(tl[g])
            out.append(acc)
        return np.asarray(out)

    results = []
    for i in range(plan.n_inputs):
        per_q = []
        for j in range(plan.n_questions[i]):
            home = plan.question_home[(i, j)]
            if plan.searched[i][j]:
                per_q.append(None)
                continue
            lp = question_lp(home)
            p, residual = option_stats(lp)
            key = plan.passes[home[0]].questions[home[1]].key
            if key in plan.floor_home:
                flp = question_lp(plan.floor_home[key])
                fp, fres = option_stats(flp)
            else:
                flp = np.full_like(lp, np.nan)
                fp = np.full_like(lp, np.nan)
                fres = np.nan
            per_q.append({"lp": lp, "p": p, "residual": residual,
                          "floor_lp": flp, "floor_p": fp, "floor_residual": fres})
        results.append(per_q)
    return results


def collect_extract(plan, top_tok_per_pass, top_lp_per_pass):
    """Per searched slot, in question order (input by input): ``(tokens[k], logprobs[k])``.

    ``top_*_per_pass[p]`` hold pass ``p``'s answers in its extraction order.
    """
    out = []
    for i in range(plan.n_inputs):
        for j in range(plan.n_questions[i]):
            if not plan.searched[i][j]:
                continue
            p, idx = plan.question_home[(i, j)]
            x = plan.passes[p].questions[idx].extract
            out.append((np.asarray(top_tok_per_pass[p][x]), np.asarray(top_lp_per_pass[p][x], dtype=np.float64)))
    return out
