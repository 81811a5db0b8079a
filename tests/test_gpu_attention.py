"""GPU parity of the branch-attention kernel against the fp64 oracle.

Tolerance: max |O_gpu - O_oracle| <= 2e-2 (bf16 output, fp32 accumulation,
bf16 probabilities in the PV product).  Packing invariance and determinism are
checked bit for bit.
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pass_values, run_attention, sample_rows
from oracle import attention as oa
from synth import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _check(lay, o, q, k, v, shape, rows, window=0):
    ref = oa.attention_rows(lay, q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                            shape.n_q_heads, shape.n_kv_heads, rows, window=window)
    got = o[torch.as_tensor(rows, device=o.device)].float().cpu().numpy()
    err = np.abs(got - ref).max()
    assert err <= TOL, err
    return err


def test_tiny_every_row(spinf):
    inputs, shape = wl.tiny(), wl.TINY
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
    o = run_attention(spinf, plan, 0, q, k, v, shape)
    _check(lay, o, q, k, v, shape, list(range(lay.T)))


# one per kernel arrangement: one CTA per head (d 64; d 128 with odd groups; d 256 with groups
# other than two), cta_group::2 pairs (d 128, even groups), two query heads stacked per CTA on
# 64-row Q tiles (d 256, groups of two)
SHAPES = [wl.Shape(4, 2, 64, 256, 1000), wl.Shape(8, 8, 128, 256, 1000), wl.Shape(40, 8, 128, 256, 1000),
          wl.Shape(8, 2, 128, 256, 1000), wl.Shape(16, 8, 256, 256, 1000), wl.Shape(6, 2, 256, 256, 1000)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"h{s.n_q_heads}-{s.n_kv_heads}-d{s.d_head}")
def test_multi_tile_trie_every_row(spinf, shape):
    inputs = wl.stress(n_questions=24, content_tokens=300, vocab=1000) + wl.tiny(vocab=1000)
    P = oracle_plan(inputs, token_budget=1024, vocab=1000)
    plan = spinf.Plan(inputs, token_budget=1024, vocab=1000)
    assert len(P.passes) >= 2
    for p in (0, len(P.passes) - 1):
        lay = P.passes[p]
        q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
        o = run_attention(spinf, plan, p, q, k, v, shape)
        _check(lay, o, q, k, v, shape, list(range(lay.T)))


@pytest.mark.parametrize("window", [1, 9, 40, 300])
def test_window(spinf, window):
    inputs, shape = wl.stress(n_questions=10, content_tokens=200, vocab=1000), wl.Shape(4, 2, 64, 256, 1000)
    lay = oracle_plan(inputs, vocab=1000).passes[0]
    plan = spinf.Plan(inputs, vocab=1000)
    q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
    o = run_attention(spinf, plan, 0, q, k, v, shape, window=window)
    _check(lay, o, q, k, v, shape, list(range(lay.T)), window=window)


def test_wide_window_is_bitwise_no_window_and_pads_are_zero(spinf):
    inputs, shape = wl.tiny(), wl.TINY
    inputs = inputs + [([5, 6, 7], [([1, 2], [[3], [4]])])]
    lay = oracle_plan(inputs, vocab=1024).passes[0]
    plan = spinf.Plan(inputs, vocab=1024)
    q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
    a = run_attention(spinf, plan, 0, q, k, v, shape)
    b = run_attention(spinf, plan, 0, q, k, v, shape, window=int(lay.pos.max()) + 1)
    c = run_attention(spinf, plan, 0, q, k, v, shape)
    assert torch.equal(a, b) and torch.equal(a, c)
    assert lay.T < lay.T_pad
    assert torch.count_nonzero(a[lay.T:]).item() == 0


def _unit_rows(lay, source):
    u = next(u for u in lay.units if u.source == source)
    return u.start, u.size


@pytest.mark.parametrize("shape", [wl.Shape(4, 2, 64, 256, 1000), wl.Shape(8, 8, 128, 256, 1000),
                                   wl.Shape(8, 2, 128, 256, 1000), wl.Shape(16, 8, 256, 256, 1000),
                                   wl.Shape(6, 2, 256, 256, 1000)],
                         ids=["d64-single", "d128-single", "d128-cg2", "d256-stacked", "d256-single"])
@pytest.mark.parametrize("window", [0, 100], ids=["no-window", "window-100"])
def test_packing_invariance_bitwise(spinf, shape, window):
    """The target's rows alone-ish and at five offsets among short inputs are bit-identical, with
    no window and with a window that bites on its 230-token content."""
    target = wl.stress(n_questions=12, content_tokens=230, vocab=1000)[0]
    others = wl.short_inputs(vocab=1000, n=40)
    outs = []
    for offset in (0, 1, 7, 17, 33):
        inputs = others[:offset] + [target] + others[offset:]
        lay = oracle_plan(inputs, vocab=1000, floors=False).passes[0]
        plan = spinf.Plan(inputs, vocab=1000, floors=False)
        q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
        o = run_attention(spinf, plan, 0, q, k, v, shape, window=window)
        s, n = _unit_rows(lay, offset)
        outs.append((s, o[s:s + n].clone()))
        if offset == 7 and window:   # the windowed rows against the oracle too
            rows = list(range(s, s + n, 7))
            _check(lay, o, q, k, v, shape, rows, window=window)
    starts = {s % 128 for s, _ in outs}
    assert len(starts) > 2
    for s, o in outs[1:]:
        assert torch.equal(o, outs[0][1]), s


@pytest.mark.parametrize("p,n_rows", [(0, 4096), (1, 2048)], ids=["pass0-contents", "pass1-floors"])
def test_wikinews_full_pass_sampled_rows(spinf, p, n_rows):
    """A share of every laid-out input of the pass (pass 0: 14 contents; pass 1: 10 contents
    and the 56 floors), each input's first and last rows, and the scoring rows."""
    f, shape = wl.WORKLOADS["wikinews"]
    inputs = f()
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[p]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
    o = run_attention(spinf, plan, p, q, k, v, shape)
    rows = sample_rows(lay, n_rows, p)
    assert len(rows) >= n_rows
    _check(lay, o, q, k, v, shape, rows)
    assert not torch.isnan(o[:lay.T]).any()


@pytest.mark.parametrize("shape", [wl.Shape(4, 2, 64, 256, 1000), wl.Shape(16, 8, 256, 256, 1000),
                                   wl.Shape(6, 2, 256, 256, 1000)], ids=["d64", "d256-stacked", "d256-single"])
def test_deep_tries_every_row(spinf, shape):
    """Rows whose root path has more than four runs take the key-by-key mask; the rest the
    per-row runs: both against the oracle on every row."""
    opts = [[1, 2, 5, 5, 5], [1, 3, 2, 5, 5], [1, 3, 3, 2, 5], [1, 3, 3, 3, 2]]
    inputs = [([7, 8, 9] * 50, [([4, 4], opts), ([6], opts)]), ([], [([2, 3], opts)])] + wl.tiny(vocab=1000)
    lay = oracle_plan(inputs, vocab=1000).passes[0]
    plan = spinf.Plan(inputs, vocab=1000)
    assert (plan.pass_info(0).row_runs[:, 0] == -1).any()
    q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
    o = run_attention(spinf, plan, 0, q, k, v, shape)
    _check(lay, o, q, k, v, shape, list(range(lay.T)))
