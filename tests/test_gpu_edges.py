"""Edge cases of the GPU path against the oracle.

* the smallest request: one content of one token, one question, two single-token
  options (two scoring rows with its floor);
* a pass of exactly 16,384 tokens (the token budget: no pad rows at all);
* options of the maximal 5 tokens (the man page's option-token limit), scored
  through their option-trie rows;
* vocabularies smaller than one 256-token tile (100) and one token past a tile (257);
* a question at the 1000-option limit, and one of 1000 two-token options (1000 trie rows);
* a content at the 4096-token limit with a question at the 256-token limit, with and without
  a window that bites.
"""
import numpy as np
import pytest

from gpu_util import oracle_plan, pass_values, run_attention, run_score, sample_rows
from oracle import attention as oa
from oracle import collect as oc
from oracle import score as osc
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu


def _attn(lay, o, q, k, v, shape, rows):
    ref = oa.attention_rows(lay, q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                            shape.n_q_heads, shape.n_kv_heads, rows)
    return float(np.abs(o[rows].float().cpu().numpy() - ref).max())


def _score(lay, h, w, lse, tlp):
    rl, rt = osc.score_rows(h.float().cpu().numpy()[lay.slot_row], lay.gather_m, lay.gather_tok,
                            w=w.float().numpy())
    return float(np.abs(lse - rl).max()), float(np.abs(tlp - rt).max()), rt


@pytest.mark.parametrize("d_head", [64, 256])
def test_smallest_request(spinf, d_head):
    shape = wl.Shape(4, 2, d_head, 256, 1000)
    inputs = [([7], [([3, 4, 5], [[10], [11]])])]
    P = oracle_plan(inputs, vocab=1000)
    plan = spinf.Plan(inputs, vocab=1000)
    lay = P.passes[0]
    assert lay.T == 1 + 3 + 3 and len(lay.slot_row) == 2   # the input and its floor
    q, k, v, h = pass_values(lay, shape)
    o = run_attention(spinf, plan, 0, q, k, v, shape)
    assert _attn(lay, o, q, k, v, shape, list(range(lay.T))) <= 2e-2
    assert float(o[lay.T:].float().abs().max()) == 0.0   # pad rows are written as zeros
    w = sv.lm_head(1000, 256)
    lse, tlp, _ = run_score(spinf, plan, 0, h, w.cuda(), None, spinf.DTYPE_BF16, shape)
    el, et, rt = _score(lay, h, w, lse, tlp)
    assert el <= 2e-3 and et <= 2e-3
    res = plan.collect([tlp])
    want = oc.collect(P, [rt])[0][0]
    assert np.abs(res["option_p"] - want["p"]).max() <= 4e-3


def test_pass_of_exactly_the_token_budget(spinf):
    """Inputs sized so that the first pass holds exactly 16,384 rows: T = T_pad, no pad row."""
    shape = wl.GEMMA
    g = np.random.default_rng(9)
    q_tmpl = [([int(x) for x in g.integers(0, 1000, 10)], [[1], [2]])]
    # each input: content + one question of 10 tokens = content + 10 rows
    sizes = [500] * 32 + [16384 - 32 * 510 - 10]
    inputs = [([int(x) for x in g.integers(0, 1000, n)], q_tmpl) for n in sizes]
    P = oracle_plan(inputs, vocab=1000, floors=False)
    lay = P.passes[0]
    assert lay.T == 16384 == lay.T_pad
    plan = spinf.Plan(inputs, vocab=1000, floors=False)
    q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
    o = run_attention(spinf, plan, 0, q, k, v, shape)
    rows = sorted(set(range(0, lay.T, 97)) | {0, lay.T - 1, lay.T - 11, 16383 - 64})
    assert _attn(lay, o, q, k, v, shape, rows) <= 2e-2


def test_five_token_options_scored(spinf):
    shape = wl.Shape(4, 2, 64, 256, 1000)
    opts = [[5, 6, 7, 8, 9], [5, 6, 7, 8, 10], [5, 11, 12, 13, 14], [15, 16, 17, 18, 19]]
    inputs = [([1, 2, 3] * 20, [([4, 4, 4], opts)]), ([21, 22], [([4, 4, 4], opts), ([30], [[31], [32, 33, 34, 35, 36]])])]
    P = oracle_plan(inputs, vocab=1000)
    plan = spinf.Plan(inputs, vocab=1000)
    w = sv.lm_head(1000, 256)
    lps, ref = [], []
    for p, lay in enumerate(P.passes):
        q, k, v, h = pass_values(lay, shape)
        lse, tlp, _ = run_score(spinf, plan, p, h, w.cuda(), None, spinf.DTYPE_BF16, shape)
        el, et, rt = _score(lay, h, w, lse, tlp)
        assert el <= 2e-3 and et <= 2e-3
        lps.append(tlp)
        ref.append(rt)
    res = plan.collect(lps)
    want = np.concatenate([r["lp"] for per_q in oc.collect(P, ref) for r in per_q])
    assert res["option_lp"].shape == (4 + 4 + 2,)
    assert np.abs(res["option_lp"] - want).max() <= 5 * 2e-3   # five token lps summed


@pytest.mark.parametrize("vocab", [100, 257])
def test_small_and_ragged_vocabularies(spinf, vocab):
    shape = wl.Shape(4, 2, 64, 256, vocab)
    inputs = wl.tiny(vocab=vocab)
    P = oracle_plan(inputs, vocab=vocab)
    plan = spinf.Plan(inputs, vocab=vocab)
    w = sv.lm_head(vocab, 256)
    for p, lay in enumerate(P.passes):
        _, _, _, h = pass_values(lay, shape)
        lse, tlp, _ = run_score(spinf, plan, p, h, w.cuda(), None, spinf.DTYPE_BF16, shape)
        el, et, _ = _score(lay, h, w, lse, tlp)
        assert el <= 2e-3 and et <= 2e-3


def test_thousand_options(spinf):
    """A question at the option limit (1000 single-token options) and one of 1000 two-token
    options (1000 option-trie rows): scores and option p against the oracle."""
    shape = wl.Shape(4, 2, 64, 256, 4096)
    g = np.random.default_rng(11)
    single = [[int(t)] for t in g.choice(4096, size=1000, replace=False)]
    firsts = g.choice(4096, size=1000, replace=False)
    double = [[int(a), int(g.integers(0, 4096))] for a in firsts]
    inputs = [([int(x) for x in g.integers(0, 4096, 120)], [([5, 6, 7], single), ([8, 9], double)])]
    P = oracle_plan(inputs, vocab=4096)
    plan = spinf.Plan(inputs, vocab=4096)
    w = sv.lm_head(4096, 256)
    lps, ref = [], []
    for p, lay in enumerate(P.passes):
        _, _, _, h = pass_values(lay, shape)
        lse, tlp, _ = run_score(spinf, plan, p, h, w.cuda(), None, spinf.DTYPE_BF16, shape)
        el, et, rt = _score(lay, h, w, lse, tlp)
        assert el <= 2e-3 and et <= 2e-3
        lps.append(tlp)
        ref.append(rt)
    res = plan.collect(lps)
    want = oc.collect(P, ref)[0]
    assert res["option_p"].shape == (2000,)
    assert np.abs(res["option_p"] - np.concatenate([want[0]["p"], want[1]["p"]])).max() <= 4e-3
    assert np.abs(res["residual"] - np.array([want[0]["residual"], want[1]["residual"]])).max() <= 4e-3


@pytest.mark.parametrize("d_head", [128, 256])
def test_longest_content_and_question(spinf, d_head):
    """A content at the 4096-token limit with a question at the 256-token limit, with and
    without a window that bites: sampled rows of every part against the oracle."""
    shape = wl.Shape(8, 4 if d_head == 256 else 2, d_head, 256, 1000)
    g = np.random.default_rng(12)
    inputs = [([int(x) for x in g.integers(0, 1000, 4096)],
               [([int(x) for x in g.integers(0, 1000, 256)], [[1], [2, 3]]), ([4, 5], [[6], [7]])])]
    P = oracle_plan(inputs, vocab=1000)
    plan = spinf.Plan(inputs, vocab=1000)
    lay = P.passes[0]
    q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
    rows = sample_rows(lay, 160, 4)
    for window in (0, 1024):
        o = run_attention(spinf, plan, 0, q, k, v, shape, window=window)
        ref = oa.attention_rows(lay, q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                                shape.n_q_heads, shape.n_kv_heads, rows, window=window)
        assert float(np.abs(o[rows].float().cpu().numpy() - ref).max()) <= 2e-2
