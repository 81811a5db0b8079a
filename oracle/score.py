"""Oracle slot scoring in fp64 (TEST INFRASTRUCTURE ONLY).

Restates "spinf-serve 0.1.1" (PyPI), "What it does": at the slot (where the
template ends) the model's next-token distribution is read for each option;
the engine returns each option's log-probability.  The man page
(PARAMETERS, ``--lm-head``) gives fp32 output of the lm head as the default.

For every scoring row ``r`` (a slot or an option-prefix row, see
:mod:`oracle.plan`):

* ``z_r[v] = sum_d h[r, d] * W[v, d]`` over the whole vocabulary, in fp64 over
  the exact input values (for fp8 weights ``W[v, d] = e4m3(code) * s_w[v]``,
  and the hidden row is first replaced by its per-row e4m3 quantisation, see
  :func:`oracle.fp8.quantize_rows`);
* ``lse_r = log sum_v exp(z_r[v])``;
* the log-probability of option token ``t`` read at row ``r`` is
  ``z_r[t] - lse_r``.

A searched slot (``{*}``, ``{n}``, ``{$}``; PyPI page, "What it does": the
most likely answers with their probabilities) reads the same distribution at
its slot row and returns the ``k`` tokens of the allowed set with the largest
``z`` (ties: the lower token id first), each with ``z - lse`` over the whole
vocabulary.
"""
from __future__ import annotations

import numpy as np

from . import fp8


def logits(h_rows, w_rows):
    """``z = h @ W^T`` in fp64."""
    return np.asarray(h_rows, dtype=np.float64) @ np.asarray(w_rows, dtype=np.float64).T


def logsumexp(z):
    """``log sum exp`` along the last axis, shifted by the maximum for range."""
    m = np.max(z, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(z - m), axis=-1, keepdims=True)))[..., 0]


def hidden_rows(h_slot, act_fp8):
    """The scoring rows as the contraction sees them (fp64).

    ``h_slot``: ``[M, D]`` values exactly representable in fp32 (bf16 inputs).
    With ``act_fp8`` the rows are quantised per row to e4m3 and rescaled.
    """
    if not act_fp8:
        return np.asarray(h_slot, dtype=np.float64)
    codes, s = fp8.quantize_rows(h_slot)
    return fp8.decode(codes) * s.astype(np.float64)[:, None]


def weight_rows(w, w_codes=None, w_scale=None, rows=slice(None)):
    """lm-head rows in fp64: bf16 values, or e4m3 codes times their row scale."""
    if w_codes is None:
        return np.asarray(w[rows], dtype=np.float64)
    return fp8.decode(w_codes[rows]) * np.asarray(w_scale[rows], dtype=np.float64)[:, None]


def score_rows(h_slot, gather_m, gather_tok, w=None, w_codes=None, w_scale=None, chunk=16384):
    """``(lse[M], token_logprob[G])`` in fp64 for one pass.

    The vocabulary is read in slices of ``chunk`` rows only to bound host memory:
    each ``z_r[v]`` is the same plain dot product whichever slice holds ``v``,
    and ``lse`` is taken once over the assembled full row.
    """
    act_fp8 = w_codes is not None
    h = hidden_rows(h_slot, act_fp8)
    V = (w if w is not None else w_codes).shape[0]
    z = np.empty((h.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, chunk):
        z[:, v0:v0 + chunk] = logits(h, weight_rows(w, w_codes, w_scale, slice(v0, v0 + chunk)))
    lse = logsumexp(z)
    gm = np.asarray(gather_m, dtype=np.int64)
    gt = np.asarray(gather_tok, dtype=np.int64)
    return lse, z[gm, gt] - lse[gm]


def topk_allowed(z_row, lse_row, allowed, k):
    """The searched-slot answer of one row: ``(tokens[k], logprobs[k])``.

    ``allowed``: a boolean mask over the vocabulary, or None for every token.
    The allowed tokens are ordered by ``z`` descending, then by token id, and the
    first ``k`` are kept; missing places (fewer than ``k`` allowed tokens) are
    ``(-1, -inf)``.
    """
    z_row = np.asarray(z_row, dtype=np.float64)
    cand = np.arange(z_row.shape[0]) if allowed is None else np.flatnonzero(np.asarray(allowed, dtype=bool))
    order = np.lexsort((cand, -z_row[cand]))      # primary key: -z; secondary: token id
    top = cand[order[:k]]
    tok = np.full(k, -1, dtype=np.int64)
    lp = np.full(k, -np.inf)
    tok[:len(top)] = top
    lp[:len(top)] = z_row[top] - lse_row
    return tok, lp


def extract_rows(h_x, x_set, token_sets, k, w=None, w_codes=None, w_scale=None, chunk=16384):
    """Searched-slot answers for the rows ``h_x`` (``[X, D]``): ``(tokens[X, k], logprobs[X, k])``.

    ``x_set[x]`` names the allowed set of row ``x`` (an index into ``token_sets``,
    boolean masks over the vocabulary), ``-1`` for every token.
    """
    act_fp8 = w_codes is not None
    h = hidden_rows(h_x, act_fp8)
    V = (w if w is not None else w_codes).shape[0]
    z = np.empty((h.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, chunk):
        z[:, v0:v0 + chunk] = logits(h, weight_rows(w, w_codes, w_scale, slice(v0, v0 + chunk)))
    lse = logsumexp(z)
    toks = np.full((h.shape[0], k), -1, dtype=np.int64)
    lps = np.full((h.shape[0], k), -np.inf)
    for x in range(h.shape[0]):
        s = int(x_set[x])
        toks[x], lps[x] = topk_allowed(z[x], lse[x], None if s < 0 else token_sets[s], k)
    return toks, lps
