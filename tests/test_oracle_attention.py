"""Pins of the oracle attention.

* Brute force: every branch endpoint recomputed as an independent, unpacked
  causal sequence (content + template + option prefix), with values drawn for
  that plain sequence and textbook causal softmax attention over it.
* Special cases: one visible key gives that key's value; a zero query gives the
  mean of the visible values; a window of 1 gives the row's own value; a window
  at least the deepest path changes nothing.
* Packing order: an input's outputs are bitwise the same alone and packed.
"""
import math

import numpy as np
import pytest

from oracle import attention as oa
from oracle import plan as op
from synth import values as sv
from synth import workloads as wl


def _textbook_causal(q, k, v, Hq, Hkv, scale):
    """Plain causal attention over a sequence [n, H, d]; returns the last row [Hq, d]."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    n = q.shape[0]
    out = np.zeros((Hq, q.shape[2]))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = scale * np.einsum("d,nd->n", q[n - 1, h], k[:, g])
        p = np.exp(s - s.max())
        p /= p.sum()
        out[h] = np.einsum("n,nd->d", p, v[:, g])
    return out


def _values(keys, T_pad, shape):
    q, k, v = sv.qkv(keys, T_pad, shape.n_q_heads, shape.n_kv_heads, shape.d_head)
    return q.float().numpy(), k.float().numpy(), v.float().numpy()


@pytest.mark.parametrize("inputs_fn", [
    lambda: wl.tiny(),
    lambda: wl.stress(n_questions=6, content_tokens=40, vocab=1024),
])
def test_brute_force_unpacked_sequences(inputs_fn):
    shape = wl.TINY
    inputs = inputs_fn()
    P = op.plan(inputs, vocab=1024)
    scale = 1.0 / math.sqrt(shape.d_head)
    checked = 0
    for lay in P.passes:
        keys = sv.path_keys(lay.tok, lay.parent, lay.T)
        q, k, v = _values(keys, lay.T_pad, shape)
        for rec in lay.questions:
            if rec.source >= 0:
                unit = next(u for u in lay.units if u.source == rec.source and rec.qidx in u.qidx)
                template, options = inputs[rec.source][1][rec.qidx]
            else:
                unit = next(u for u in lay.units if u.source < 0 and u.floor_key == rec.key)
                template, options = rec.key
            for o, gs in zip(options, rec.option_gather):
                for i, g in enumerate(gs):
                    seq = list(unit.content) + list(template) + list(o[:i])
                    sk = sv.seq_keys(seq)
                    bq, bk, bv = _values(sk, len(seq), shape)
                    want = _textbook_causal(bq, bk, bv, shape.n_q_heads, shape.n_kv_heads, scale)
                    row = int(lay.slot_row[lay.gather_m[g]])
                    got = oa.attention_rows(lay, q, k, v, shape.n_q_heads, shape.n_kv_heads, [row])[0]
                    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
                    checked += 1
        # content rows too: a content row is a causal prefix of its content
        for u in lay.units:
            for i in range(0, len(u.content), 7):
                seq = list(u.content[: i + 1])
                bq, bk, bv = _values(sv.seq_keys(seq), len(seq), shape)
                want = _textbook_causal(bq, bk, bv, shape.n_q_heads, shape.n_kv_heads, scale)
                got = oa.attention_rows(lay, q, k, v, shape.n_q_heads, shape.n_kv_heads, [u.start + i])[0]
                np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    assert checked > 0


def _tiny_layout():
    inputs = wl.tiny()
    P = op.plan(inputs, vocab=1024)
    lay = P.passes[0]
    keys = sv.path_keys(lay.tok, lay.parent, lay.T)
    return lay, _values(keys, lay.T_pad, wl.TINY)


def test_single_visible_key_returns_its_value():
    lay, (q, k, v) = _tiny_layout()
    first_rows = [u.start for u in lay.units if len(u.content) > 0]
    got = oa.attention_rows(lay, q, k, v, 4, 2, first_rows)
    for i, r in enumerate(first_rows):
        for h in range(4):
            np.testing.assert_array_equal(got[i, h], v[r, h // 2])


def test_zero_query_gives_mean_of_visible_values():
    lay, (q, k, v) = _tiny_layout()
    q0 = np.zeros_like(q)
    rows = list(range(0, lay.T, 5))
    got = oa.attention_rows(lay, q0, k, v, 4, 2, rows)
    for i, r in enumerate(rows):
        vis = lay.visible(r)
        for h in range(4):
            np.testing.assert_allclose(got[i, h], v[vis, h // 2].astype(np.float64).mean(0), atol=1e-12)


def test_window_one_is_self_and_wide_window_is_none():
    lay, (q, k, v) = _tiny_layout()
    rows = list(range(lay.T))
    w1 = oa.attention_rows(lay, q, k, v, 4, 2, rows, window=1)
    for i, r in enumerate(rows):
        for h in range(4):
            np.testing.assert_array_equal(w1[i, h], v[r, h // 2])
    wide = oa.attention_rows(lay, q, k, v, 4, 2, rows, window=int(lay.pos.max()) + 1)
    none = oa.attention_rows(lay, q, k, v, 4, 2, rows)
    np.testing.assert_array_equal(wide, none)
    narrow = oa.attention_rows(lay, q, k, v, 4, 2, rows, window=16)
    assert not np.array_equal(narrow, none)


def test_window_keeps_the_last_w_keys_of_the_path():
    lay, (q, k, v) = _tiny_layout()
    W = 9
    r = int(lay.slot_row[0])
    path = lay.visible(r)
    kept = path[-W:]
    scale = 1 / 8
    got = oa.attention_rows(lay, q, k, v, 4, 2, [r], window=W)[0]
    for h in range(4):
        s = scale * (k[kept, h // 2].astype(np.float64) @ q[r, h].astype(np.float64))
        p = np.exp(s - s.max())
        np.testing.assert_allclose(got[h], p @ v[kept, h // 2] / p.sum(), atol=1e-12)


def test_packing_order_is_bitwise_invisible():
    inputs = wl.tiny()
    alone = op.plan([inputs[1]], floors=False).passes[0]
    packed = op.plan(inputs, floors=False).passes[0]
    ua, up = alone.units[0], next(u for u in packed.units if u.source == 1)
    outs = []
    for lay, u in ((alone, ua), (packed, up)):
        keys = sv.path_keys(lay.tok, lay.parent, lay.T)
        q, k, v = _values(keys, lay.T_pad, wl.TINY)
        outs.append(oa.attention_rows(lay, q, k, v, 4, 2, list(range(u.start, u.start + u.size))))
    np.testing.assert_array_equal(outs[0], outs[1])
