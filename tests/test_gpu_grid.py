"""A placeholder-grid request end to end on the GPU.

"spinf-serve 0.1.1" (PyPI page, "What it does"): placeholders turn one template
into a grid of questions.  A grid is planned as one question per combination of
its placeholder values (first placeholder slowest), each an ordinary question of
its input laid out exactly like the same question written out by hand.  So:

* the cells' option log-probabilities match the oracle's on the same layout
  (2e-3 nats, bf16 lm head) and the attention rows of the pass match it within
  the attention tolerance (2e-2);
* every output of the grid request -- attention rows, row log-sum-exps, token
  log-probabilities and the collected p / residual / floor -- is bit-identical to
  that of the request with the cells written out as questions.
"""
import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pass_values, run_attention, run_score
from oracle import attention as oa
from oracle import collect as oc
from oracle import plan as op
from oracle import score as osc
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu


def _request(vocab, seed=3):
    g = np.random.default_rng(seed)
    ids = lambda n: [int(x) for x in g.integers(0, vocab, size=n)]  # noqa: E731
    inputs = []
    for c in range(3):
        own = [(ids(9), [[t] for t in g.choice(vocab, 2, replace=False).tolist()])]
        # 3 values x 2 values, literal pieces around them; multi-token option on the second grid
        grid_a = ([ids(4), ids(2), ids(3)], [[ids(1), ids(2), ids(3)], [ids(2), ids(1)]],
                  [[t] for t in g.choice(vocab, 3, replace=False).tolist()])
        t = g.choice(vocab, 3, replace=False).tolist()
        grid_b = ([ids(5), ids(1)], [[ids(3), ids(1)]], [[t[0], t[1]], [t[2]]])
        inputs.append((ids(int(g.integers(40, 150))), own, [grid_a, grid_b]))
    written = [(content, own + [(c[0], c[1]) for gr in grids for c in op.expand_grid(gr)])
               for content, own, grids in inputs]
    return inputs, written


def _run(spinf, inputs, shape, w):
    P = oracle_plan(inputs, vocab=shape.vocab)
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    outs, lps = [], []
    for p, lay in enumerate(P.passes):
        q, k, v, h = pass_values(lay, shape)
        o = run_attention(spinf, plan, p, q, k, v, shape)
        lse, tlp, _ = run_score(spinf, plan, p, h, w, None, spinf.DTYPE_BF16, shape)
        outs.append((lay, q, k, v, h, o, lse, tlp))
        lps.append(tlp)
    return P, plan, outs, plan.collect(lps)


@pytest.mark.parametrize("d_head", [64, 256])
def test_grid_request_matches_oracle_and_written_out_questions(spinf, d_head):
    shape = wl.Shape(4, 2, d_head, 256, 1024)
    inputs, written = _request(shape.vocab)
    w = sv.lm_head(shape.vocab, shape.d_model)
    wd = w.cuda()
    P, plan, outs, res = _run(spinf, inputs, shape, wd)
    assert sum(P.n_questions) == 3 * (1 + 6 + 2)
    ref_lp = []
    for lay, q, k, v, h, o, lse, tlp in outs:
        ref = oa.attention_rows(lay, q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                                shape.n_q_heads, shape.n_kv_heads, list(range(lay.T)))
        assert np.abs(o[:lay.T].float().cpu().numpy() - ref).max() <= 2e-2
        rl, rt = osc.score_rows(h.float().cpu().numpy()[lay.slot_row], lay.gather_m, lay.gather_tok,
                                w=w.float().numpy())
        assert np.abs(lse - rl).max() <= 2e-3
        assert np.abs(tlp - rt).max() <= 2e-3
        ref_lp.append(tlp)
    # the collect over the GPU's token lps against the oracle's collect over the same lps
    want = oc.collect(P, ref_lp)
    want_lp = np.concatenate([r["lp"] for per_q in want for r in per_q])
    assert np.abs(res["option_lp"] - want_lp).max() <= 1e-12
    # bit-identical to the written-out request
    P2, plan2, outs2, res2 = _run(spinf, written, shape, wd)
    assert len(outs2) == len(outs)
    for a, b in zip(outs, outs2):
        assert torch.equal(a[5], b[5])                            # attention, every row
        assert np.array_equal(a[6], b[6]) and np.array_equal(a[7], b[7])
    for key in ("option_lp", "option_p", "option_floor_lp", "option_floor_p", "residual", "floor_residual"):
        assert np.array_equal(res[key], res2[key]), key
