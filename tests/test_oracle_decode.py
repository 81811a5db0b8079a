"""Pins of the decode-step oracle: a decode row equals (1) textbook causal attention over
the unpacked sequence content + template + decoded tokens, and (2) the packed oracle
when the decoded tokens are written into the template and the request is planned again."""
import math

import numpy as np

from oracle import attention as oa
from oracle import decode as od
from oracle import plan as op
from synth import values as sv
from synth import workloads as wl


def _setup(seed=0):
    inputs = [([5, 6, 7, 8], [([9, 10], [[11], [12]]), ([13, 14, 15], None, -1)]),
              ([20, 21], [([22], None, -1), ([23, 24], [[25]])])]
    P = op.plan(inputs, floors=False)
    lay = P.passes[0]
    anchors = [int(lay.slot_row[m]) for m in lay.x_m]          # the searched slots' rows
    # two steps: each slot decodes a first token, then the first slot a second one
    toks = [(0, -1, 101), (1, -1, 202), (0, 0, 103)]          # (slot, parent decode row, token)
    anchor = np.array([anchors[s] for s, _, _ in toks])
    parent = np.array([p for _, p, _ in toks])
    return inputs, lay, anchor, parent, toks


def _decode_values(lay, anchor, parent, toks, shape):
    """Path keys of the decode rows (their tokens continue the anchor's path)."""
    keys_pass = sv.path_keys(lay.tok, lay.parent, lay.T)
    keys = []
    for r, (_, p, t) in enumerate(toks):
        base = keys_pass[anchor[r]] if p < 0 else keys[p]
        keys.append(sv.extend_key(base, t))
    q, k, v = sv.qkv(keys, len(keys), shape.n_q_heads, shape.n_kv_heads, shape.d_head)
    return keys_pass, keys, q.double().numpy(), k.double().numpy(), v.double().numpy()


def test_decode_rows_equal_unpacked_causal_attention():
    shape = wl.TINY
    inputs, lay, anchor, parent, toks = _setup()
    keys_pass, keys, qd, kd, vd = _decode_values(lay, anchor, parent, toks, shape)
    qp, kp, vp = (t.double().numpy() for t in sv.qkv(keys_pass, lay.T_pad, shape.n_q_heads, shape.n_kv_heads,
                                                        shape.d_head))
    got = od.decode_attention(lay, qd, kp, vp, kd, vd, anchor, parent, list(range(len(toks))), shape.n_q_heads,
                              shape.n_kv_heads)
    # the same rows as plain sequences: content + template + decoded tokens, values from their own keys
    searched = [(i, q) for i, (_, qs) in enumerate(inputs) for q in qs if q[1] is None]
    scale = 1.0 / math.sqrt(shape.d_head)
    for r, (s, p, t) in enumerate(toks):
        i, (template, _, _) = searched[s]
        dec = [toks[c][2] for c in od.chain(parent, r)]
        seq = list(inputs[i][0]) + list(template) + dec
        sk = sv.seq_keys(seq)
        q, k, v = (x.double().numpy() for x in sv.qkv(sk, len(seq), shape.n_q_heads, shape.n_kv_heads,
                                                      shape.d_head))
        for h in range(shape.n_q_heads):
            g = h * shape.n_kv_heads // shape.n_q_heads
            sc = scale * (k[:, g] @ q[-1, h])
            w = np.exp(sc - sc.max())
            np.testing.assert_allclose(got[r, h], (w @ v[:, g]) / w.sum(), rtol=0, atol=1e-12)


def test_decode_rows_equal_replanned_template():
    shape = wl.TINY
    inputs, lay, anchor, parent, toks = _setup()
    keys_pass, keys, qd, kd, vd = _decode_values(lay, anchor, parent, toks, shape)
    qp, kp, vp = (t.double().numpy() for t in sv.qkv(keys_pass, lay.T_pad, shape.n_q_heads, shape.n_kv_heads,
                                                        shape.d_head))
    got = od.decode_attention(lay, qd[[2]], kp, vp, kd, vd, anchor, parent, [2], shape.n_q_heads, shape.n_kv_heads)
    # slot 0 with both decoded tokens written into its template
    ext = [(inputs[0][0], [inputs[0][1][0], ([13, 14, 15, 101, 103], None, -1)]), inputs[1]]
    lay2 = op.plan(ext, floors=False).passes[0]
    k2 = sv.path_keys(lay2.tok, lay2.parent, lay2.T)
    q2, kk2, v2 = (t.double().numpy() for t in sv.qkv(k2, lay2.T_pad, shape.n_q_heads, shape.n_kv_heads,
                                                       shape.d_head))
    row = int(lay2.slot_row[lay2.x_m[0]])        # the extended template's last row
    want = oa.attention_rows(lay2, q2, kk2, v2, shape.n_q_heads, shape.n_kv_heads, [row])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_chain_order():
    parent = np.array([-1, -1, 0, 2, 1])
    assert od.chain(parent, 3) == [0, 2, 3] and od.chain(parent, 4) == [1, 4] and od.chain(parent, 1) == [1]
