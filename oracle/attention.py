"""Oracle tree-masked attention in fp64 (TEST INFRASTRUCTURE ONLY).

Restates "spinf-serve 0.1.1" (PyPI), "What it does" and "Speed and scale":
each question is a branch of one pass; a branch token attends to its own
content and causally to its own branch, never to a sibling branch or to another
packed input.  In the oracle the visible keys of a row are its root path, taken
from :meth:`oracle.plan.PassLayout.visible`.

Readings (the pages give no formula):

* softmax attention with scale ``1/sqrt(d_head)`` unless one is given, no
  logit soft-capping;
* grouped heads: query head ``h`` reads key/value head ``h * Hkv // Hq``;
* an optional window ``W``: key ``k`` stays visible to row ``q`` only while
  ``pos[q] - pos[k] < W`` (``W`` counts the row itself); ``W = 0`` means none.
"""
from __future__ import annotations

import math

import numpy as np


def attention_rows(layout, q, k, v, n_q_heads, n_kv_heads, rows, scale=None, window=0):
    """Attention output for the given packed rows, every head, in fp64.

    ``q``: ``[T_pad, Hq, d]``, ``k``/``v``: ``[T_pad, Hkv, d]`` (any float dtype;
    converted to fp64).  Returns ``[len(rows), Hq, d]`` fp64.
    """
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((len(rows), n_q_heads, d), dtype=np.float64)
    for i, row in enumerate(rows):
        keys = np.asarray(layout.visible(int(row)), dtype=np.int64)
        if window:
            keys = keys[layout.pos[row] - layout.pos[keys] < window]
        for h in range(n_q_heads):
            g = h * n_kv_heads // n_q_heads
            qv = np.asarray(q[row, h], dtype=np.float64)
            kk = np.asarray(k[keys, g], dtype=np.float64)
            vv = np.asarray(v[keys, g], dtype=np.float64)
            s = scale * (kk @ qv)
            w = np.exp(s - s.max())
            out[i, h] = (w @ vv) / w.sum()
    return out


def real_rows(layout):
    """Rows that belong to an input (pad rows excluded)."""
    return np.arange(layout.T, dtype=np.int64)
