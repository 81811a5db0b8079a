"""Oracle of the decoding steps of searched slots in fp64 (TEST INFRASTRUCTURE ONLY).

Restates "spinf-serve 0.1.1" (PyPI), "What it does" and "Speed and scale":
extraction slots ({*} text, {n} numbers, {$} amounts) are decoded on the same read
of the content: the content and the questions are not read again, the slots of
many inputs are decoded together.

Reading (the pages give no algorithm): a decode row extends the root path of a row
of a packed pass (a searched slot's last template row, its *anchor*) by tokens
chosen at earlier steps.  Its visible keys are the anchor's visible keys in the
pass (the cached keys and values of the pass, not recomputed), then the decode
rows of its own chain from the first decoded token down to itself.  Attention over
them is the same softmax as in :mod:`oracle.attention`.  So a decode row's output
equals that of the same tokens laid out in a pass as the question's template
continued by the decoded tokens.

Decode rows are described by two arrays over all decode rows so far:
``anchor[r]`` (a pass row) and ``parent[r]`` (an earlier decode row of the same
chain, or -1 for the first decoded token, whose parent is the anchor itself).
"""
from __future__ import annotations

import math

import numpy as np


def chain(parent, r):
    """Decode rows from the first decoded token of ``r``'s chain down to ``r``."""
    out = []
    while r >= 0:
        out.append(int(r))
        r = int(parent[r])
    return out[::-1]


def decode_attention(layout, q_dec, k_pass, v_pass, k_dec, v_dec, anchor, parent, rows, n_q_heads, n_kv_heads,
                     scale=None):
    """Outputs ``[len(rows), Hq, d]`` (fp64) of the decode rows ``rows``.

    ``q_dec``: ``[len(rows), Hq, d]`` (the queries of those rows, in order);
    ``k_pass``/``v_pass``: the pass's ``[T_pad, Hkv, d]``; ``k_dec``/``v_dec``:
    ``[n_dec, Hkv, d]`` of every decode row.
    """
    d = q_dec.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((len(rows), n_q_heads, d))
    for i, r in enumerate(rows):
        pk = np.asarray(layout.visible(int(anchor[r])), dtype=np.int64)
        ck = np.asarray(chain(parent, r), dtype=np.int64)
        for h in range(n_q_heads):
            g = h * n_kv_heads // n_q_heads
            kk = np.concatenate([np.asarray(k_pass[pk, g], np.float64), np.asarray(k_dec[ck, g], np.float64)])
            vv = np.concatenate([np.asarray(v_pass[pk, g], np.float64), np.asarray(v_dec[ck, g], np.float64)])
            s = scale * (kk @ np.asarray(q_dec[i, h], np.float64))
            w = np.exp(s - s.max())
            out[i, h] = (w @ vv) / w.sum()
    return out
