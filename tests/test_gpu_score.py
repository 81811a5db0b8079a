"""GPU parity of slot scoring (gather + lm head + full-vocabulary lse + option lps).

Tolerances against the fp64 oracle: 2e-3 nats with bf16 weights, 2e-2 with e4m3
weights (the oracle applies the same per-row e4m3 quantisation to the hidden
rows, which is compared bit for bit).
"""
import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pass_values, run_score
from oracle import fp8
from oracle import score as osc
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu


def _oracle(lay, hidden, w=None, codes=None, scale=None, rows=None):
    h = hidden.float().cpu().numpy()[lay.slot_row]
    gm, gt = lay.gather_m, lay.gather_tok
    if rows is not None:
        sel = np.isin(gm, rows)
        remap = {m: i for i, m in enumerate(rows)}
        gm2 = np.array([remap[m] for m in gm[sel]], dtype=np.int64)
        lse, lp = osc.score_rows(h[rows], gm2, gt[sel], w=w, w_codes=codes, w_scale=scale)
        return lse, lp, sel
    lse, lp = osc.score_rows(h, gm, gt, w=w, w_codes=codes, w_scale=scale)
    return lse, lp, None


@pytest.mark.parametrize("workload", ["tiny", "trie"])
def test_bf16_every_row(spinf, workload):
    if workload == "tiny":
        inputs, shape = wl.tiny(), wl.TINY
    else:   # M > 128 over several slot tiles, multi-token options, ragged vocabulary (1000 = 3 x 256 + 232)
        inputs, shape = wl.stress(n_questions=80, content_tokens=100, vocab=1000), wl.Shape(4, 2, 64, 512, 1000)
    P = oracle_plan(inputs, vocab=shape.vocab)
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    w = sv.lm_head(shape.vocab, shape.d_model)
    for p, lay in enumerate(P.passes):
        _, _, _, h = pass_values(lay, shape)
        lse, tlp, _ = run_score(spinf, plan, p, h, w.cuda(), None, spinf.DTYPE_BF16, shape)
        rl, rt, _ = _oracle(lay, h, w=w.float().numpy())
        assert np.abs(lse - rl).max() <= 2e-3
        assert np.abs(tlp - rt).max() <= 2e-3
        if workload == "trie":
            assert lay.slot_row.size > 128


def test_e4m3_every_row_and_codes(spinf):
    inputs, shape = wl.stress(n_questions=40, content_tokens=100, vocab=1000), wl.Shape(4, 2, 64, 512, 1000)
    P = oracle_plan(inputs, vocab=shape.vocab)
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    w = sv.lm_head(shape.vocab, shape.d_model)
    codes, scale = sv.e4m3_rows(w)
    lay = P.passes[0]
    _, _, _, h = pass_values(lay, shape)
    lse, tlp, ws = run_score(spinf, plan, 0, h, codes.cuda(), scale.cuda(), spinf.DTYPE_E4M3, shape)
    rl, rt, _ = _oracle(lay, h, codes=codes.numpy(), scale=scale.numpy())
    assert np.abs(lse - rl).max() <= 2e-2
    assert np.abs(tlp - rt).max() <= 2e-2
    # the quantised hidden rows the kernel used are the oracle's, bit for bit
    M = lay.slot_row.size
    want_codes, want_scale = fp8.quantize_rows(h.float().cpu().numpy()[lay.slot_row])
    got_codes = ws[: M * shape.d_model].view(M, shape.d_model).cpu().numpy()
    np.testing.assert_array_equal(got_codes, want_codes)


def test_gemma_full_vocab_sampled_rows(spinf):
    f, shape = wl.WORKLOADS["wikinews"]
    inputs = f()
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    _, _, _, h = pass_values(lay, shape)
    w = sv.lm_head(shape.vocab, shape.d_model, device="cuda")
    lse, tlp, _ = run_score(spinf, plan, 0, h, w, None, spinf.DTYPE_BF16, shape)
    rows = list(range(0, lay.slot_row.size, 37))[:24] + [lay.slot_row.size - 1]
    rl, rt, sel = _oracle(lay, h, w=w.cpu().float().numpy(), rows=rows)
    assert np.abs(lse[rows] - rl).max() <= 2e-3
    assert np.abs(tlp[sel] - rt).max() <= 2e-3
    assert np.isfinite(lse).all() and np.isfinite(tlp).all()


def test_scores_do_not_depend_on_other_rows(spinf):
    shape = wl.Shape(4, 2, 64, 512, 1000)
    target = wl.stress(n_questions=30, content_tokens=50, vocab=1000)[0]
    others = wl.short_inputs(vocab=1000, n=60)
    w = sv.lm_head(shape.vocab, shape.d_model).cuda()
    results = []
    for offset in (0, 13, 60):
        inputs = others[:offset] + [target] + others[offset:]
        lay = oracle_plan(inputs, vocab=1000, floors=False).passes[0]
        plan = spinf.Plan(inputs, vocab=1000, floors=False)
        _, _, _, h = pass_values(lay, shape)
        lse, tlp, _ = run_score(spinf, plan, 0, h, w, None, spinf.DTYPE_BF16, shape)
        rec = [r for r in lay.questions if r.source == offset]
        gs = [g for r in rec for gg in r.option_gather for g in gg]
        ms = sorted({int(lay.gather_m[g]) for g in gs})
        results.append((lse[ms], tlp[gs]))
    for lse_i, tlp_i in results[1:]:
        assert np.array_equal(lse_i, results[0][0]) and np.array_equal(tlp_i, results[0][1])
