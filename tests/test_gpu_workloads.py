"""GPU parity at the full sizes of the benchmark workloads, on sampled rows, and
batch invariance of the target input across ten random packings.

* moderation-shaped pass (Gemma-class heads): attention with and without the
  1024-token window (which never bites at these depths, so both must be
  bitwise equal), bf16 scoring;
* many-questions stress pass (Qwen-class heads, d_head 128, 40/8 heads,
  vocabulary 151936, d_model 5120): attention with and without a window that
  bites (content of 4000 tokens), scoring of multi-token options;
* batch invariance: a 470-token content with 56 questions, alone (twice) and
  inserted at a random index among 2000 short inputs (10 packings); its attention
  rows and its e4m3 scores must be bit-identical in every run.
"""
import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pass_values, run_attention, run_score, sample_rows
from oracle import attention as oa
from oracle import score as osc
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu


def _attn_check(lay, o, q, k, v, shape, rows, window=0):
    ref = oa.attention_rows(lay, q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                            shape.n_q_heads, shape.n_kv_heads, rows, window=window)
    got = o[torch.as_tensor(rows, device=o.device)].float().cpu().numpy()
    err = float(np.abs(got - ref).max())
    assert err <= 2e-2, err


def _score_check(lay, h, w, lse, tlp, n_rows=12):
    rows = list(range(0, len(lay.slot_row), max(1, len(lay.slot_row) // n_rows)))
    hs = h.float().cpu().numpy()[lay.slot_row]
    sel = np.isin(lay.gather_m, rows)
    remap = {m: i for i, m in enumerate(rows)}
    gm = np.array([remap[m] for m in lay.gather_m[sel]], dtype=np.int64)

    class Rows:   # bf16 rows converted on demand (bounded host memory)
        shape = tuple(w.shape)

        def __getitem__(self, sl):
            return w[sl].float().cpu().numpy()

    rl, rt = osc.score_rows(hs[rows], gm, lay.gather_tok[sel], w=Rows())
    assert np.abs(lse[rows] - rl).max() <= 2e-3
    assert np.abs(tlp[sel] - rt).max() <= 2e-3


def test_moderation_pass_windowed_and_scores(spinf):
    f, shape = wl.WORKLOADS["moderation"]
    inputs = f()
    P = oracle_plan(inputs, vocab=shape.vocab)
    assert len(P.passes) == 3
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    lay = P.passes[0]
    q, k, v, h = pass_values(lay, shape)
    o = run_attention(spinf, plan, 0, q, k, v, shape)
    ow = run_attention(spinf, plan, 0, q, k, v, shape, window=shape.window)
    assert int(lay.pos[:lay.T].max()) < shape.window and torch.equal(o, ow)
    _attn_check(lay, o, q, k, v, shape, sample_rows(lay, 4096, 1))   # a share of every message of the pass
    w = sv.lm_head(shape.vocab, shape.d_model, device="cuda")
    lse, tlp, _ = run_score(spinf, plan, 0, h, w, None, spinf.DTYPE_BF16, shape)
    _score_check(lay, h, w, lse, tlp)


def test_stress_pass_qwen_shapes(spinf):
    f, shape = wl.WORKLOADS["stress"]
    inputs = f()
    P = oracle_plan(inputs, vocab=shape.vocab)
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    lay = P.passes[0]
    q, k, v, h = pass_values(lay, shape)
    rows = sample_rows(lay, 512, 2)   # 40 heads over ~4,000-key paths: the oracle's cost bounds the sample
    o = run_attention(spinf, plan, 0, q, k, v, shape)
    _attn_check(lay, o, q, k, v, shape, rows)
    ow = run_attention(spinf, plan, 0, q, k, v, shape, window=shape.window)
    _attn_check(lay, ow, q, k, v, shape, rows, window=shape.window)
    assert not torch.equal(o, ow)          # the window bites on a 4000-token content
    w = sv.lm_head(shape.vocab, shape.d_model, device="cuda")
    lse, tlp, _ = run_score(spinf, plan, 0, h, w, None, spinf.DTYPE_BF16, shape)
    _score_check(lay, h, w, lse, tlp)


def test_batch_invariance_ten_packings_e4m3(spinf):
    shape = wl.GEMMA
    w = sv.lm_head(shape.vocab, shape.d_model, device="cuda")
    codes, scale = sv.e4m3_rows(w)
    del w
    target = wl.invariance_target()
    # alone twice (a difference there would be a race, not an order dependence), then ten packings
    runs = [([target], 0), ([target], 0)] + [wl.invariance_packing(s) for s in range(1, 11)]
    ref = None
    offsets = set()
    for inputs, idx in runs:
        P = oracle_plan(inputs, vocab=shape.vocab)
        p, u = next((p, u) for p, lay in enumerate(P.passes) for u in lay.units if u.source == idx)
        lay = P.passes[p]
        plan = spinf.Plan(inputs, vocab=shape.vocab)
        q, k, v, h = pass_values(lay, shape)
        o = run_attention(spinf, plan, p, q, k, v, shape)
        lse, tlp, _ = run_score(spinf, plan, p, h, codes, scale, spinf.DTYPE_E4M3, shape)
        recs = [r for r in lay.questions if r.source == idx]
        gs = [g for r in recs for gg in r.option_gather for g in gg]
        ms = sorted({int(lay.gather_m[g]) for g in gs})
        got = (o[u.start:u.start + u.size].cpu(), lse[ms], tlp[gs])
        offsets.add(u.start % 128)
        if ref is None:
            ref = got
            continue
        assert torch.equal(got[0], ref[0])
        assert np.array_equal(got[1], ref[1]) and np.array_equal(got[2], ref[2])
    assert len(offsets) > 3
