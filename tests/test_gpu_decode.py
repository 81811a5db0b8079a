"""GPU parity of the decoding steps of searched slots: decode-row attention on the pass's
cached keys and values (spinf_decode_attention) and next-token answers at those rows
(spinf_score_rows), against the fp64 oracle, against the packed kernels on the request
planned again with the decoded tokens in the template, and for batch invariance."""
import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pack_token_sets, pass_values, run_attention, run_score_extract
from oracle import decode as od
from oracle import score as osc
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


SHAPES = {"d64": wl.TINY, "d128": wl.Shape(40, 8, 128, 512, 1000), "d256": wl.Shape(16, 8, 256, 512, 1000)}
# head groupings of the decode kernel's row blocks: 8 rows of 1 head, 2 rows of 4 heads, 1 row of 8 heads
GROUPS = {"d128-g1": wl.Shape(8, 8, 128, 512, 1000), "d256-g4": wl.Shape(16, 4, 256, 512, 1000),
          "d64-g8": wl.Shape(64, 8, 64, 512, 1000)}


def _request(vocab):
    base = wl.stress(n_questions=8, content_tokens=90, vocab=vocab) + wl.tiny(vocab=vocab)
    return wl.with_searched_slots(base, 2, vocab=vocab)


def _decode_rows(lay, vocab, seed=0):
    """Two decoding steps: a first token for every searched slot, a second for every other one.
    Returns (anchor, parent, tokens) over all decode rows."""
    g = np.random.default_rng(seed)
    anchors = [int(lay.slot_row[m]) for m in lay.x_m]
    anchor, parent, toks = [], [], []
    for a in anchors:
        anchor.append(a)
        parent.append(-1)
        toks.append(int(g.integers(0, vocab)))
    for s in range(0, len(anchors), 2):
        anchor.append(anchors[s])
        parent.append(s)
        toks.append(int(g.integers(0, vocab)))
    return np.array(anchor), np.array(parent), toks


def _values(lay, anchor, parent, toks, shape):
    kp = sv.path_keys(lay.tok, lay.parent, lay.T)
    keys = []
    for r, t in enumerate(toks):
        keys.append(sv.extend_key(kp[anchor[r]] if parent[r] < 0 else keys[parent[r]], t))
    q, k, v = sv.qkv(keys, len(keys), shape.n_q_heads, shape.n_kv_heads, shape.d_head)
    return kp, keys, q, k, v


@pytest.mark.parametrize("name", list(SHAPES) + list(GROUPS))
def test_decode_matches_oracle(spinf, name):
    shape = {**SHAPES, **GROUPS}[name]
    inputs = _request(shape.vocab)
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    plan.upload(0)
    anchor, parent, toks = _decode_rows(lay, shape.vocab)
    _, _, qd, kd, vd = _values(lay, anchor, parent, toks, shape)
    qp, kp, vp, _ = pass_values(lay, shape, hidden_rows=False)
    rows = list(range(len(toks)))[::-1]            # any order of the step's rows
    q = qd[rows].contiguous().cuda()
    o = torch.full_like(q, float("nan"))
    spinf.decode_attention(plan, 0, q, kp, vp, kd.cuda(), vd.cuda(), _i32(anchor), _i32(parent), _i32(rows), o,
                           shape.n_q_heads, shape.n_kv_heads, shape.d_head)
    plan.device_status()
    want = od.decode_attention(lay, qd[rows].double().numpy(), kp.double().cpu().numpy(), vp.double().cpu().numpy(),
                               kd.double().numpy(), vd.double().numpy(), anchor, parent, rows, shape.n_q_heads,
                               shape.n_kv_heads)
    assert np.abs(o.float().cpu().numpy() - want).max() <= 2e-2


def test_decode_equals_replanned_branch_attention(spinf):
    """The decode rows of one slot against the packed attention kernel on the request planned
    again with those tokens written into the slot's template."""
    shape = SHAPES["d128"]
    inputs = _request(shape.vocab)
    lay = oracle_plan(inputs, vocab=shape.vocab, floors=False).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab, floors=False)
    plan.upload(0)
    anchor, parent, toks = _decode_rows(lay, shape.vocab)
    _, _, qd, kd, vd = _values(lay, anchor, parent, toks, shape)
    qp, kp, vp, _ = pass_values(lay, shape, hidden_rows=False)
    r2 = len(lay.x_m)                               # the second token of slot 0
    o = torch.empty(2, shape.n_q_heads, shape.d_head, dtype=torch.bfloat16, device="cuda")
    spinf.decode_attention(plan, 0, qd[[0, r2]].contiguous().cuda(), kp, vp, kd.cuda(), vd.cuda(), _i32(anchor),
                           _i32(parent), _i32([0, r2]), o, shape.n_q_heads, shape.n_kv_heads, shape.d_head)
    plan.device_status()
    # slot 0 is the first searched question of input 0: write both tokens into its template
    i0 = next(i for i, (_, qs) in enumerate(inputs) if any(q[1] is None for q in qs))
    qs = list(inputs[i0][1])
    j0 = next(j for j, q in enumerate(qs) if q[1] is None)
    qs[j0] = (list(qs[j0][0]) + [toks[0], toks[r2]], None, qs[j0][2])
    ext = list(inputs)
    ext[i0] = (inputs[i0][0], qs)
    lay2 = oracle_plan(ext, vocab=shape.vocab, floors=False).passes[0]
    plan2 = spinf.Plan(ext, vocab=shape.vocab, floors=False)
    q2, k2, v2, _ = pass_values(lay2, shape, hidden_rows=False)
    o2 = run_attention(spinf, plan2, 0, q2, k2, v2, shape)
    last = int(lay2.slot_row[lay2.x_m[0]])
    got = o.float().cpu().numpy()
    want = o2[[last - 1, last]].float().cpu().numpy()
    assert np.abs(got - want).max() <= 2e-2


def test_decode_rows_do_not_depend_on_the_step(spinf):
    shape = SHAPES["d256"]
    inputs = _request(shape.vocab)
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    plan.upload(0)
    anchor, parent, toks = _decode_rows(lay, shape.vocab)
    _, _, qd, kd, vd = _values(lay, anchor, parent, toks, shape)
    qp, kp, vp, _ = pass_values(lay, shape, hidden_rows=False)
    rows = list(range(len(toks)))
    o_all = torch.empty(len(rows), shape.n_q_heads, shape.d_head, dtype=torch.bfloat16, device="cuda")
    spinf.decode_attention(plan, 0, qd.cuda(), kp, vp, kd.cuda(), vd.cuda(), _i32(anchor), _i32(parent), _i32(rows),
                           o_all, shape.n_q_heads, shape.n_kv_heads, shape.d_head)
    for r in (0, len(rows) - 1):
        o1 = torch.empty(1, shape.n_q_heads, shape.d_head, dtype=torch.bfloat16, device="cuda")
        spinf.decode_attention(plan, 0, qd[[r]].contiguous().cuda(), kp, vp, kd.cuda(), vd.cuda(), _i32(anchor),
                               _i32(parent), _i32([r]), o1, shape.n_q_heads, shape.n_kv_heads, shape.d_head)
        plan.device_status()
        assert torch.equal(o1[0], o_all[r])


@pytest.mark.parametrize("name", list(SHAPES) + list(GROUPS))
def test_beam_rows_share_their_anchor_and_match_alone(spinf, name):
    """Beam layout: four decode rows per searched slot next to each other (first tokens), then
    four second tokens each extending one of them.  Rows of one anchor are computed together;
    each row equals, bit for bit, the same row computed alone, and the oracle."""
    shape = {**SHAPES, **GROUPS}[name]
    inputs = _request(shape.vocab)
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    plan.upload(0)
    g = np.random.default_rng(3)
    anchors = [int(lay.slot_row[m]) for m in lay.x_m]
    anchor, parent, toks = [], [], []
    for a in anchors:                       # step 1: beam of 4 first tokens per slot
        for _ in range(4):
            anchor.append(a)
            parent.append(-1)
            toks.append(int(g.integers(0, shape.vocab)))
    n1 = len(toks)
    for s in range(len(anchors)):           # step 2: each beam extends one of its first tokens
        for b in range(4):
            anchor.append(anchors[s])
            parent.append(4 * s + int(g.integers(0, 4)))
            toks.append(int(g.integers(0, shape.vocab)))
    anchor, parent = np.array(anchor), np.array(parent)
    _, _, qd, kd, vd = _values(lay, anchor, parent, toks, shape)
    qp, kp, vp, _ = pass_values(lay, shape, hidden_rows=False)
    kd, vd = kd.cuda(), vd.cuda()
    for rows in (list(range(n1)), list(range(n1, len(toks)))):
        q = qd[rows].contiguous().cuda()
        o = torch.full_like(q, float("nan"))
        spinf.decode_attention(plan, 0, q, kp, vp, kd, vd, _i32(anchor), _i32(parent), _i32(rows), o,
                               shape.n_q_heads, shape.n_kv_heads, shape.d_head)
        plan.device_status()
        want = od.decode_attention(lay, qd[rows].double().numpy(), kp.double().cpu().numpy(),
                                   vp.double().cpu().numpy(), kd.double().cpu().numpy(), vd.double().cpu().numpy(),
                                   anchor, parent, rows, shape.n_q_heads, shape.n_kv_heads)
        assert np.abs(o.float().cpu().numpy() - want).max() <= 2e-2
        for j in (0, 1, 5, len(rows) - 1):
            o1 = torch.empty(1, shape.n_q_heads, shape.d_head, dtype=torch.bfloat16, device="cuda")
            spinf.decode_attention(plan, 0, qd[[rows[j]]].contiguous().cuda(), kp, vp, kd, vd, _i32(anchor),
                                   _i32(parent), _i32([rows[j]]), o1, shape.n_q_heads, shape.n_kv_heads,
                                   shape.d_head)
            plan.device_status()
            assert torch.equal(o1[0], o[j])


def test_decode_checks_rows_on_the_device(spinf):
    """A bad row (parent not earlier, a chain of 70 tokens, q_row out of range) is written as
    zeros and reported as SPINF_E_DEVICE_CHECK; the good rows of the same call are unaffected."""
    shape = wl.TINY
    inputs = _request(shape.vocab)
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    plan.upload(0)
    a = int(lay.slot_row[lay.x_m[0]])
    qp, kp, vp, _ = pass_values(lay, shape, hidden_rows=False)
    g = torch.Generator().manual_seed(1)
    kv = torch.randn(72, 2, 64, generator=g).to(torch.bfloat16).cuda()
    q = torch.randn(2, 4, 64, generator=g).to(torch.bfloat16).cuda()
    cases = [([a, a], [-1, 1], [0, 1]),                              # row 1's parent is itself
             ([a] * 70, [-1] + list(range(69)), [0, 69]),            # row 69's chain has 70 tokens
             ([a, a], [-1, 0], [0, 5])]                              # q_row 5 does not exist
    good = None
    for anchor, parent, rows in cases:
        o = torch.full_like(q, float("nan"))
        spinf.decode_attention(plan, 0, q, kp, vp, kv, kv, _i32(anchor), _i32(parent), _i32(rows), o, 4, 2, 64)
        with pytest.raises(spinf.SpinfError) as e:
            plan.device_status()
        assert e.value.status_name == "DEVICE_CHECK"
        assert torch.count_nonzero(o[1]).item() == 0 and torch.isfinite(o[0]).all()
        good = o[0].clone() if good is None else good
        assert torch.equal(o[0], good)   # row 0 (one token on the anchor) is the same each time


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_score_rows_equal_searched_slot_answers(spinf, dtype):
    """Answers at caller-given rows equal, bit for bit, the searched-slot answers of the same
    hidden rows scored inside a pass (a row's answer depends on its own values only), and
    match the oracle."""
    shape = wl.Shape(4, 2, 64, 512, 1000)
    inputs = _request(shape.vocab)
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab, extract_k=12)
    sets = wl.token_sets(shape.vocab, n_sets=2, density=0.02)
    w = sv.lm_head(shape.vocab, shape.d_model)
    wk = {"bf16": (w.cuda(), None, spinf.DTYPE_BF16)}
    if dtype == "e4m3":
        codes, scale = sv.e4m3_rows(w)
        wk["e4m3"] = (codes.cuda(), scale.cuda(), spinf.DTYPE_E4M3)
    wd, ws, wt = wk[dtype]
    _, _, _, h = pass_values(lay, shape)
    _, _, tt, tl = run_score_extract(spinf, plan, 0, h, wd, ws, wt, shape, sets)
    rows = h[torch.as_tensor(lay.slot_row[lay.x_m], dtype=torch.long)].contiguous()
    n, k = rows.shape[0], 12
    lse = torch.empty(n, device="cuda")
    top_tok = torch.empty(n, k, dtype=torch.int32, device="cuda")
    top_lp = torch.empty(n, k, device="cuda")
    spinf.score_rows(plan, rows, wd, ws, wt, shape.d_model, shape.vocab, k, lse, top_tok, top_lp,
                     token_set=_i32(lay.x_set), token_sets=pack_token_sets(sets).cuda())
    plan.device_status()
    assert np.array_equal(top_tok.cpu().numpy(), tt) and np.array_equal(top_lp.cpu().numpy(), tl)
    if dtype == "bf16":
        ot, ol = osc.extract_rows(rows.float().cpu().numpy(), lay.x_set, sets, k, w=w.float().numpy())
        z = osc.logits(rows.float().cpu().numpy(), w.float().numpy())
        got = top_tok.cpu().numpy()
        for x in range(n):
            for j in range(k):
                assert got[x, j] == ot[x, j] or abs(z[x, got[x, j]] - z[x, ot[x, j]]) <= 2e-3
        fin = ot >= 0
        assert np.abs(top_lp.cpu().numpy()[fin] - ol[fin]).max() <= 2e-3
