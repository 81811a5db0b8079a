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

The fp8 linears of the calibrated scheme (man page, DESCRIPTION and PARAMETERS
``--quant``: ``fp8s``, scores bit-identical alone or packed) use static scales, fixed
before the request: one per activation tensor (``x_scale``) and one per weight output
channel (``w_scale[out]``).  Reading: the activation codes are
``e4m3(x / x_scale)`` (fp32 division, round to nearest even, saturating at 448) and
``y = (codes_x * x_scale) @ (codes_w * w_scale[:, None]).T``.  A static scale makes a
row's codes a function of the row alone, whatever else is in the batch.
"""
from __future__ import annotations

import numpy as np

from . import attention
from . import fp8


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


def qkv_rope(x, w_qkv, pos, n_q_heads, n_kv_heads, d_head, theta):
    """q, k (turned at tree depth) and v of the packed rows, fp64: the projection
    ``x @ w_qkv.T`` split into heads, then :func:`rope` on q and k."""
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w_qkv, dtype=np.float64).T
    q, k, v = split_qkv(y, n_q_heads, n_kv_heads, d_head)
    return rope(q, pos, theta), rope(k, pos, theta), v


def quantize_static(x, x_scale):
    """e4m3 codes of ``x`` with a static scale: ``e4m3(x / x_scale)``, the division in fp32."""
    scaled = (np.asarray(x, dtype=np.float32) / np.float32(x_scale)).astype(np.float32)
    return fp8.encode_rne_sat(scaled)


def linear_fp8(x_codes, x_scale, w_codes, w_scale):
    """``(codes_x * x_scale) @ (codes_w * w_scale[:, None]).T`` in fp64."""
    xs = fp8.decode(x_codes) * float(np.float32(x_scale))
    ws = fp8.decode(w_codes) * np.asarray(w_scale, dtype=np.float64)[:, None]
    return xs @ ws.T
