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


def test_gemma_full_vocab_e4m3_sampled_rows(spinf):
    """The e4m3 lm head at the Gemma-class size (vocabulary 262144, d_model 3840) on the
    Wikinews-shaped pass 0: per-row-scaled weights ("spinf-serve" man page, DESCRIPTION, the
    fp8s scheme; PARAMETERS, --lm-head f32out), against the oracle's e4m3 scoring within
    2e-2 nats on 25 slot rows spread over the pass and every gathered token of those rows;
    the quantised hidden rows the kernel used equal the oracle's bit for bit."""
    f, shape = wl.WORKLOADS["wikinews"]
    inputs = f()
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    _, _, _, h = pass_values(lay, shape)
    codes, scale = sv.e4m3_rows(sv.lm_head(shape.vocab, shape.d_model, device="cuda"))
    lse, tlp, ws = run_score(spinf, plan, 0, h, codes, scale, spinf.DTYPE_E4M3, shape)
    M = lay.slot_row.size
    rows = list(range(0, M, 33))[:24] + [M - 1]
    assert len(rows) >= 12
    rl, rt, sel = _oracle(lay, h, codes=codes.cpu().numpy(), scale=scale.cpu().numpy(), rows=rows)
    assert sel.sum() >= len(rows)            # every option token read at those rows
    assert np.abs(lse[rows] - rl).max() <= 2e-2
    assert np.abs(tlp[sel] - rt).max() <= 2e-2
    assert np.isfinite(lse).all() and np.isfinite(tlp).all()
    want_codes, _ = fp8.quantize_rows(h.float().cpu().numpy()[lay.slot_row])
    got_codes = ws[: M * shape.d_model].view(M, shape.d_model).cpu().numpy()
    np.testing.assert_array_equal(got_codes, want_codes)


def _score_passes(spinf, plan, passes, hs, w, w_scale, w_dtype, shape, slot_rows=False):
    infos = [plan.pass_info(p) for p in passes]
    for p in passes:
        plan.upload(p)
    ws = torch.empty(spinf.score_passes_workspace_bytes(plan, passes, shape.vocab, shape.d_model, w_dtype),
                     dtype=torch.uint8, device="cuda")
    lse = [torch.full((max(i.M, 1),), float("nan"), device="cuda") for i in infos]
    tlp = [torch.full((max(i.G, 1),), float("nan"), device="cuda") for i in infos]
    spinf.score_passes(plan, passes, hs, w, w_scale, w_dtype, shape.d_model, shape.vocab, lse, tlp, ws,
                       slot_rows=slot_rows)
    plan.device_status()
    torch.cuda.synchronize()
    return [(l[:i.M].cpu().numpy(), t[:i.G].cpu().numpy()) for l, t, i in zip(lse, tlp, infos)]


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
def test_score_passes_bitwise_equals_per_pass_calls(spinf, fp8):
    """Several passes in one lm-head sweep (spinf_score_passes): every row's lse and every token
    log-probability bit-identical to the one-pass calls, whatever the order the passes are
    listed in and whichever passes share the call; ragged vocabulary (1000 = 3 x 256 + 232),
    multi-token options, passes whose row counts are not multiples of 128."""
    shape = wl.Shape(4, 2, 64, 512, 1000)
    inputs = wl.stress(n_questions=120, content_tokens=300, vocab=1000)
    P = oracle_plan(inputs, vocab=1000, token_budget=1024)
    plan = spinf.Plan(inputs, vocab=1000, token_budget=1024)
    n = len(P.passes)
    assert n >= 4 and any(len(lay.slot_row) % 128 for lay in P.passes)
    w = sv.lm_head(shape.vocab, shape.d_model)
    w_scale = None
    w_dtype = spinf.DTYPE_E4M3 if fp8 else spinf.DTYPE_BF16
    if fp8:
        w, w_scale = sv.e4m3_rows(w)
        w_scale = w_scale.cuda()
    w = w.cuda()
    hs = {p: pass_values(lay, shape)[3] for p, lay in enumerate(P.passes)}
    ref = {p: run_score(spinf, plan, p, hs[p], w, w_scale, w_dtype, shape)[:2] for p in range(n)}
    for passes in (list(range(n)), list(reversed(range(n))), [n - 1, 0], [1]):
        got = _score_passes(spinf, plan, passes, [hs[p] for p in passes], w, w_scale, w_dtype, shape)
        for p, (lse, tlp) in zip(passes, got):
            assert np.array_equal(lse, ref[p][0]) and np.array_equal(tlp, ref[p][1]), (passes, p)
    # the hidden states of the scoring rows only, compacted in scoring-row order
    slots = [hs[p][torch.as_tensor(lay.slot_row, device="cuda").long()].contiguous() for p, lay in enumerate(P.passes)]
    got = _score_passes(spinf, plan, list(range(n)), slots, w, w_scale, w_dtype, shape, slot_rows=True)
    for p, (lse, tlp) in enumerate(got):
        assert np.array_equal(lse, ref[p][0]) and np.array_equal(tlp, ref[p][1]), ("slot rows", p)


def test_score_passes_wikinews_job_one_sweep(spinf):
    """Both passes of the Wikinews-shaped job at Gemma-class sizes in one call: bit-identical to
    the one-pass calls, and within 2e-3 nats of the oracle on sampled rows of both passes."""
    f, shape = wl.WORKLOADS["wikinews"]
    inputs = f()
    P = oracle_plan(inputs, vocab=shape.vocab)
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    w = sv.lm_head(shape.vocab, shape.d_model, device="cuda")
    hs = [pass_values(lay, shape)[3] for lay in P.passes]
    got = _score_passes(spinf, plan, list(range(len(P.passes))), hs, w, None, spinf.DTYPE_BF16, shape)
    for p, lay in enumerate(P.passes):
        lse, tlp, _ = run_score(spinf, plan, p, hs[p], w, None, spinf.DTYPE_BF16, shape)
        assert np.array_equal(got[p][0], lse) and np.array_equal(got[p][1], tlp)
        rows = [0, len(lay.slot_row) // 2, len(lay.slot_row) - 1]
        rl, rt, sel = _oracle(lay, hs[p], w=w.cpu().float().numpy(), rows=rows)
        assert np.abs(got[p][0][rows] - rl).max() <= 2e-3
        assert np.abs(got[p][1][sel] - rt).max() <= 2e-3
