"""GPU parity of searched slots ({*} {n} {$}): the top tokens of the allowed set at a
slot row, read in the same lm-head pass as the scored options.

Against the fp64 oracle: the kernel decides the order in fp32, so its j-th token must
be the oracle's j-th token or one whose fp64 logit is within a logit tolerance of it
(a near tie); every token must be allowed and distinct; its log-probability must be
within 2e-3 nats (bf16) or 2e-2 (e4m3) of the oracle's value for that token.  With
logits that are exact in fp32 (a one-hot hidden row, small integer weights) the
tokens, ties included, must equal the oracle's exactly.
"""
import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pass_values, run_score, run_score_extract
from oracle import score as osc
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu

SMALL = wl.Shape(4, 2, 64, 512, 1000)   # ragged vocabulary: 3 x 256 + 232


def _oracle_z(h_rows, w=None, codes=None, scale=None, chunk=16384):
    """fp64 logits of the searched rows over the whole vocabulary, and their lse."""
    h = osc.hidden_rows(h_rows, codes is not None)
    V = (w if w is not None else codes).shape[0]
    z = np.empty((h.shape[0], V))
    for v0 in range(0, V, chunk):
        z[:, v0:v0 + chunk] = osc.logits(h, osc.weight_rows(w, codes, scale, slice(v0, v0 + chunk)))
    return z, osc.logsumexp(z)


def _check(lay, top_tok, top_lp, z, lse, sets, k, tol_lp, tol_z):
    for x in range(len(lay.x_m)):
        s = int(lay.x_set[x])
        allowed = np.ones(z.shape[1], bool) if s < 0 else np.asarray(sets[s], bool)
        ot, ol = osc.topk_allowed(z[x], lse[x], None if s < 0 else sets[s], k)
        kt, kl = top_tok[x], top_lp[x]
        n_valid = min(k, int(allowed.sum()))
        assert (kt[:n_valid] >= 0).all() and (kt[n_valid:] == -1).all(), x
        assert np.isneginf(kl[n_valid:]).all(), x
        v = kt[:n_valid]
        assert len(set(v.tolist())) == n_valid and allowed[v].all(), x
        assert np.abs(kl[:n_valid] - (z[x, v] - lse[x])).max(initial=0) <= tol_lp, x
        for j in range(n_valid):
            assert kt[j] == ot[j] or abs(z[x, kt[j]] - z[x, ot[j]]) <= tol_z, (x, j)
        assert np.all(np.diff(kl[:n_valid]) <= 0), x


def _searched_plan(spinf, base, n_slots, vocab, **kw):
    inputs = wl.with_searched_slots(base, n_slots, vocab=vocab)
    return inputs, oracle_plan(inputs, vocab=vocab, **kw), spinf.Plan(inputs, vocab=vocab, **kw)


@pytest.mark.parametrize("k", [1, 8, 16])
def test_exact_logits_ties_bit_exact(spinf, k):
    """One-hot hidden rows and small integer weights: every logit is exact in fp32, with
    many ties; the kernel's tokens equal the oracle's (ties by the lower id)."""
    shape = SMALL
    base = wl.tiny(vocab=shape.vocab)
    inputs, P, plan = _searched_plan(spinf, base, 6, shape.vocab, extract_k=k)
    lay = P.passes[0]
    g = np.random.default_rng(k)
    w = torch.zeros(shape.vocab, shape.d_model)
    w[:, 0] = torch.from_numpy(g.integers(-3, 4, size=shape.vocab).astype(np.float32))
    w[:, 1] = torch.from_numpy(g.integers(-2, 3, size=shape.vocab).astype(np.float32))
    w = w.to(torch.bfloat16)
    h = torch.zeros(lay.T_pad, shape.d_model)
    for i, r in enumerate(lay.slot_row.tolist()):
        h[r, 0] = 1.0 + (i % 3)
        h[r, 1] = float(i % 2)
    h = h.to(torch.bfloat16)
    sets = wl.token_sets(shape.vocab, density=0.05)
    _, _, tt, tl = run_score_extract(spinf, plan, 0, h.cuda(), w.cuda(), None, spinf.DTYPE_BF16, shape, sets)
    z, lse = _oracle_z(h.float().numpy()[lay.slot_row[lay.x_m]], w=w.float().numpy())
    ot, ol = osc.extract_rows(h.float().numpy()[lay.slot_row[lay.x_m]], lay.x_set, sets, k, w=w.float().numpy())
    np.testing.assert_array_equal(tt, ot)
    finite = ot >= 0
    assert np.abs(tl[finite] - ol[finite]).max() <= 2e-3
    assert np.isneginf(tl[~finite]).all()


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_matches_oracle_every_slot(spinf, dtype):
    """Slots over several scoring tiles (M > 128), three sets, ragged vocabulary."""
    shape = SMALL
    base = wl.stress(n_questions=70, content_tokens=100, vocab=shape.vocab)
    inputs, P, plan = _searched_plan(spinf, base, 9, shape.vocab, extract_k=12)
    lay = P.passes[0]
    assert lay.slot_row.size > 128 and len(lay.x_m) == 9
    sets = wl.token_sets(shape.vocab, n_sets=2, density=0.02)
    w = sv.lm_head(shape.vocab, shape.d_model)
    _, _, _, h = pass_values(lay, shape)
    hx = h.float().cpu().numpy()[lay.slot_row[lay.x_m]]
    if dtype == "bf16":
        lse, tlp, tt, tl = run_score_extract(spinf, plan, 0, h, w.cuda(), None, spinf.DTYPE_BF16, shape, sets)
        z, zl = _oracle_z(hx, w=w.float().numpy())
        tol = 2e-3
    else:
        codes, scale = sv.e4m3_rows(w)
        lse, tlp, tt, tl = run_score_extract(spinf, plan, 0, h, codes.cuda(), scale.cuda(), spinf.DTYPE_E4M3, shape,
                                             sets)
        z, zl = _oracle_z(hx, codes=codes.numpy(), scale=scale.numpy())
        tol = 2e-2
    _check(lay, tt, tl, z, zl, sets, 12, tol, tol)
    # the scored outputs are those of plain scoring, bit for bit
    if dtype == "bf16":
        lse0, tlp0, _ = run_score(spinf, plan, 0, h, w.cuda(), None, spinf.DTYPE_BF16, shape)
        assert np.array_equal(lse, lse0) and np.array_equal(tlp, tlp0)


def test_gemma_full_vocab(spinf):
    """The Wikinews-shaped job with two searched slots per content ({*} and {n}) at the
    full 262144-token vocabulary: every slot of pass 0 against the oracle."""
    f, shape = wl.WORKLOADS["wikinews"]
    inputs, P, plan = _searched_plan(spinf, f(), 2, shape.vocab)
    lay = P.passes[0]
    sets = wl.token_sets(shape.vocab, n_sets=1)
    _, _, _, h = pass_values(lay, shape)
    w = sv.lm_head(shape.vocab, shape.d_model, device="cuda")
    k = plan.extract_counts()[1]
    _, _, tt, tl = run_score_extract(spinf, plan, 0, h, w, None, spinf.DTYPE_BF16, shape, sets)
    hx = h.float().cpu().numpy()[lay.slot_row[lay.x_m]]
    z, zl = _oracle_z(hx, w=w.cpu().float().numpy())
    _check(lay, tt, tl, z, zl, sets, k, 2e-3, 2e-3)


def test_answers_do_not_depend_on_packing(spinf):
    shape = SMALL
    target = wl.with_searched_slots([wl.stress(n_questions=10, content_tokens=50, vocab=1000)[0]], 4,
                                    vocab=1000)[0]
    others = wl.short_inputs(vocab=1000, n=60)
    sets = wl.token_sets(1000, density=0.03)
    w = sv.lm_head(shape.vocab, shape.d_model).cuda()
    got = []
    for offset in (0, 17, 60):
        inputs = others[:offset] + [target] + others[offset:]
        lay = oracle_plan(inputs, vocab=1000).passes[0]
        plan = spinf.Plan(inputs, vocab=1000)
        _, _, _, h = pass_values(lay, shape)
        _, _, tt, tl = run_score_extract(spinf, plan, 0, h, w, None, spinf.DTYPE_BF16, shape, sets)
        xs = [r.extract for r in lay.questions if r.source == offset and r.extract >= 0]
        got.append((tt[xs], tl[xs]))
    for tt, tl in got[1:]:
        assert np.array_equal(tt, got[0][0]) and np.array_equal(tl, got[0][1])


def test_bad_token_set_rejected(spinf):
    shape = SMALL
    inputs = [([1, 2, 3], [([4, 5], None, 3)])]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    _, _, _, h = pass_values(lay, shape)
    w = sv.lm_head(shape.vocab, shape.d_model).cuda()
    with pytest.raises(spinf.SpinfError) as e:
        run_score_extract(spinf, plan, 0, h, w, None, spinf.DTYPE_BF16, shape, wl.token_sets(shape.vocab, 2))
    assert e.value.status_name == "INVALID"
