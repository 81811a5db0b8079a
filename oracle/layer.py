"""Oracle of the steps around the attention call (TEST INFRASTRUCTURE ONLY): rotary
positions at tree depth and the packed layer QKV -> rotary -> attention -> output.

Restates "spinf-serve 0.1.1" (PyPI), "What it does": every question is a branch of
one packed pass and an input's scores are the same alone or packed; the man page
DESCRIPTION speaks of one packed forward.  Readings (the pages give no formula):

* rotary embedding, rotate-half form: the pairs ``(x[i], x[i + d/2])``, ``i < d/2``,
  turn by the angle ``pos * theta ** (-2 i / d)``;
* ``pos`` is the row's depth on its own root path (the layout's ``pos``), so a
  branch token takes the position it has in its unpacked sequence;
* projections are plain products ``y = x @ w.T`` (``w`` is ``[out, in]``); the QKV
  output is the concatenation q | k | v along features.
"""
from __future__ import annotations

import numpy as np

from . import attention


def rope(x, pos, theta):
    """``x`` ``[T, H, d]`` turned by ``pos`` ``[T]`` (fp64 result)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = float(theta) ** (-2.0 * np.arange(half) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x0, x1 = x[..., :half], x[..., half:]
    return np.concatenate([x0 * c - x1 * s, x1 * c + x0 * s], axis=-1)


def split_qkv(y, n_q_heads, n_kv_heads, d_head):
    """``[T, (Hq + 2 Hkv) d]`` -> q ``[T, Hq, d]``, k, v ``[T, Hkv, d]``."""
    T = y.shape[0]
    nq, nk = n_q_heads * d_head, n_kv_heads * d_head
    return (y[:, :nq].reshape(T, n_q_heads, d_head), y[:, nq:nq + nk].reshape(T, n_kv_heads, d_head),
            y[:, nq + nk:nq + 2 * nk].reshape(T, n_kv_heads, d_head))


def packed_layer_rows(layout, x, w_qkv, w_o, n_q_heads, n_kv_heads, d_head, theta, rows):
    """Output ``[len(rows), D]`` of x -> QKV -> rotary at tree depth -> attention -> output
    projection, for the given packed rows, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    q, k, v = split_qkv(x @ np.asarray(w_qkv, dtype=np.float64).T, n_q_heads, n_kv_heads, d_head)
    q, k = rope(q, layout.pos, theta), rope(k, layout.pos, theta)
    o = attention.attention_rows(layout, q, k, v, n_q_heads, n_kv_heads, rows)
    return o.reshape(len(rows), n_q_heads * d_head) @ np.asarray(w_o, dtype=np.float64).T
