"""The product planner (C++, through the C ABI) against the oracle planner: bit-exact layouts.

Covers every workload shape, splits of long inputs, multi-token option tries,
fuzzed requests, the error statuses, and the collect step.
"""
import numpy as np
import pytest

from oracle import collect as oc
from oracle import plan as op
from synth import workloads as wl

FIELDS = ("tok", "parent", "pos", "end", "anchor", "tile_ptr", "tile_kv", "tile_len", "slot_row", "gather_m",
          "gather_tok", "x_m", "x_set")


def _compare(spinf, inputs, **opts):
    P = op.plan(inputs, **opts)
    Q = spinf.Plan(inputs, **opts)
    assert Q.num_passes == len(P.passes)
    for p, lay in enumerate(P.passes):
        info = Q.pass_info(p)
        assert (info.T, info.T_pad) == (lay.T, lay.T_pad)
        for f in FIELDS:
            a, b = getattr(info, f), getattr(lay, f)
            assert np.array_equal(a, b), (p, f)
        assert info.unit_start.tolist() == [u.start for u in lay.units] + [lay.T]
        assert info.unit_source.tolist() == [u.source for u in lay.units]
        _check_runs(info, lay)
    return P, Q


def _check_runs(info, lay, sample=512):
    """Each row's runs (the kernel's per-row mask) cover exactly the oracle's root path."""
    rows = np.arange(lay.T_pad)
    if lay.T_pad > 4096:
        g = np.random.default_rng(lay.T)
        rows = np.unique(np.concatenate([g.choice(lay.T_pad, sample, replace=False), [0, lay.T - 1, lay.T_pad - 1]]))
    for q in rows.tolist():
        want = lay.visible(q) if q < lay.T else [q]
        n_runs = 1 + sum(1 for a, b in zip(want, want[1:]) if b != a + 1)
        r = info.row_runs[q]
        if r[0] == -1:
            assert n_runs > 4, q
            continue
        got = sorted(k for i in range(4) for k in range(r[2 * i], r[2 * i + 1]))
        assert got == want, q
        assert r[1] == q + 1   # nearest run first: it ends at the row itself


@pytest.mark.parametrize("name", ["tiny", "wikinews", "moderation", "stress"])
def test_workloads_bit_exact(spinf, name):
    f, shape = wl.WORKLOADS[name]
    _compare(spinf, f(), vocab=shape.vocab)


@pytest.mark.parametrize("seed", range(1, 11))
def test_invariance_packing_bit_exact(spinf, seed):
    """Every one of the ten packings of the batch-invariance pass plans exactly like the oracle."""
    inputs, _ = wl.invariance_packing(seed)
    _compare(spinf, inputs, vocab=262144)


def test_invariance_target_alone_bit_exact(spinf):
    _compare(spinf, [wl.invariance_target()], vocab=262144)


def _target_tiles(spinf, inputs, idx, key_tile, q_rows=128):
    """Per row of the target input (relative to its first row): the executed KV tiles of
    its Q tile that hold a key the row sees, as (first key, length, visible keys), all
    relative to the input's first row; and that every other executed tile of the row's Q
    tile holds no key the row sees."""
    P = op.plan(inputs, vocab=262144)
    p, u = next((p, u) for p, lay in enumerate(P.passes) for u in lay.units if u.source == idx)
    lay = P.passes[p]
    tp, tk, tl = spinf.Plan(inputs, vocab=262144).tile_schedule(p, 0, key_tile, q_rows)
    out = []
    for r in range(u.start, u.start + u.size):
        vis = set(lay.visible(r))
        seq = []
        for e in range(tp[r // q_rows], tp[r // q_rows + 1]):
            seen = tuple(k - u.start for k in range(tk[e], tk[e] + tl[e]) if k in vis)
            if seen:
                seq.append((int(tk[e]) - u.start, int(tl[e]), seen))
        assert sum(len(t[2]) for t in seq) == len(vis), r   # every visible key is in an executed tile
        out.append(tuple(seq))
    return out, u.start


@pytest.mark.parametrize("key_tile,q_rows", [(64, 128), (128, 128), (64, 64)])
def test_invariance_target_executed_tiles(spinf, key_tile, q_rows):
    """The batch-invariance target's rows meet the same anchored KV tiles, in the same order
    and with the same visible keys at the same columns, alone and in all ten packings
    (what makes a row's attention output bit-identical alone or packed); every other
    executed tile of its Q tile is fully masked for it."""
    ref, _ = _target_tiles(spinf, [wl.invariance_target()], 0, key_tile, q_rows)
    offsets = set()
    for seed in range(1, 11):
        inputs, idx = wl.invariance_packing(seed)
        got, start = _target_tiles(spinf, inputs, idx, key_tile, q_rows)
        offsets.add(start % 128)
        assert got == ref, seed
    assert len(offsets) > 3   # the packings put the target at several offsets within a Q tile


@pytest.mark.parametrize("budget", [256, 700, 2048])
def test_splits_and_tries(spinf, budget):
    inputs = wl.stress(n_questions=60, content_tokens=150, vocab=1000)
    _compare(spinf, inputs, token_budget=budget, vocab=1000)
    _compare(spinf, inputs, token_budget=budget, floors=False, floor_prefix=[1, 2])
    _compare(spinf, inputs, token_budget=budget, floor_prefix=[5, 6, 7])


@pytest.mark.parametrize("budget", [10, 11, 12])
def test_exact_fit_stays_in_its_pass(spinf, budget):
    """Inputs of 6 and 5 tokens: one pass at budget 11 (an exact fit), two at 10 and one at 12."""
    inputs = [([1, 2, 3, 4], [([5, 6], [[7]])]), ([1, 2, 3], [([8, 9], [[7]])])]
    P, Q = _compare(spinf, inputs, token_budget=budget, floors=False)
    assert Q.num_passes == (2 if budget == 10 else 1)


def test_shared_question_lists_plan_like_separate_ones(spinf):
    """Inputs that share one question-list object (marshalled once) plan exactly like the
    same request written with separate, equal lists, and like the oracle."""
    import copy
    shared = [([5, 6, 7], [[1], [2]]), ([8, 9], [[3, 4], [3, 5]]), ([2, 2], None, 0)]
    other = [([4], [[1]])]
    empty = []
    grid = ([[1, 2], [3]], [[[7], [8, 9]]], [[1], [2]])
    inputs = [([10, 11, 12], shared), ([13] * 40, shared), ([14, 15], other), ([16], empty, [grid]),
              ([17, 18], shared), ([19], empty), ([], shared)]
    P1, Q1 = _compare(spinf, inputs, vocab=100)
    P2, Q2 = _compare(spinf, copy.deepcopy(inputs), vocab=100)
    for p in range(Q1.num_passes):
        a, b = Q1.pass_info(p), Q2.pass_info(p)
        for f in FIELDS:
            assert np.array_equal(getattr(a, f), getattr(b, f)), (p, f)


def test_floor_keys(spinf):
    """One floor per distinct (template, option lists in order): option order, option token
    splits and template length tell floors apart; equal questions in separate lists share one."""
    qs = [([1, 2], [[3], [4]]), ([1, 2], [[4], [3]]), ([1, 2], [[3, 4]]), ([1, 2], [[3], [4], [5]]),
          ([1, 2, 2], [[3], [4]]), ([1], [[2, 3], [4]]), ([1], [[2], [3, 4]])]
    inputs = [([9, 9, 9], [(list(q[0]), [list(o) for o in q[1]])]) for q in qs]   # one question each
    inputs += [([8], [(list(q[0]), [list(o) for o in q[1]]) for q in qs])]   # the same questions again
    P, Q = _compare(spinf, inputs, vocab=100)
    n_floor_units = sum(1 for lay in P.passes for u in lay.units if u.source < 0)
    assert n_floor_units == len(qs)


def test_schedule_cache_under_concurrent_callers(spinf):
    """The per-pass schedules are built on first use under the plan's lock: many threads
    asking at once (the C calls run without the interpreter lock) all get the schedule a
    single caller gets."""
    import concurrent.futures
    inputs = wl.stress(n_questions=24, content_tokens=300, vocab=1000) + wl.tiny(vocab=1000)
    ref = spinf.Plan(inputs, token_budget=1024, vocab=1000)
    keys = [(p, w, kt) for p in range(ref.num_passes) for w in (0, 7, 64) for kt in (64, 128)]
    assert len(keys) >= 12
    want = {k: ref.tile_schedule(*k) for k in keys}
    plan = spinf.Plan(inputs, token_budget=1024, vocab=1000)
    with concurrent.futures.ThreadPoolExecutor(8) as pool:
        futures = [(k, pool.submit(plan.tile_schedule, *k)) for k in keys * 6]
        for k, f in futures:
            got = f.result()
            assert all(np.array_equal(a, b) for a, b in zip(got, want[k])), k


@pytest.mark.parametrize("form", ["int64 arrays", "int32 arrays", "tuples"])
def test_token_sequences_as_arrays_or_tuples(spinf, form):
    """Contents, templates and options given as numpy arrays or tuples plan exactly like the
    same request written with lists."""
    inputs = wl.stress(n_questions=20, content_tokens=120, vocab=1000) + wl.tiny(vocab=1000)
    conv = {"int64 arrays": lambda t: np.asarray(t, dtype=np.int64),
            "int32 arrays": lambda t: np.asarray(t, dtype=np.int32), "tuples": tuple}[form]
    other = [(conv(c), [(conv(q[0]), [conv(o) for o in q[1]]) for q in qs]) for c, qs in inputs]
    a, b = spinf.Plan(inputs, vocab=1000), spinf.Plan(other, vocab=1000)
    assert a.num_passes == b.num_passes
    for p in range(a.num_passes):
        x, y = a.pass_info(p), b.pass_info(p)
        for f in FIELDS:
            assert np.array_equal(getattr(x, f), getattr(y, f)), (p, f)


def test_inputs_at_the_limits(spinf):
    """Content of 4096 tokens, a 256-token template, 1000 options, a 5-token option: accepted
    and laid out like the oracle."""
    for inp in [([1] * 4096, [([2], [[3]])]), ([1], [([2] * 256, [[3]])]),
                ([1], [([2], [[t] for t in range(1000)])]), ([1], [([2], [[3, 4, 5, 6, 7], [3]])])]:
        _compare(spinf, [inp])
    _compare(spinf, [([], [([2] * 9, [[3, 4]])])], token_budget=10)   # its floor is exactly the budget


def test_fuzzed_requests(spinf):
    g = np.random.default_rng(7)
    for trial in range(40):
        inputs = []
        for _ in range(int(g.integers(1, 12))):
            content = g.integers(0, 50, size=int(g.integers(0, 300))).tolist()
            qs = []
            for _ in range(int(g.integers(0 if content else 1, 6))):
                opts, seen = [], set()
                for _ in range(int(g.integers(1, 5))):
                    o = tuple(g.integers(0, 6, size=int(g.integers(1, 4))).tolist())
                    if o not in seen:
                        seen.add(o)
                        opts.append(list(o))
                qs.append((g.integers(0, 50, size=int(g.integers(1, 20))).tolist(), opts))
            if not content and not qs:
                content = [1]
            inputs.append((content, qs))
        budget = int(g.choice([128, 300, 1000, 16384]))
        try:
            op.plan(inputs, token_budget=budget)
        except op.PlanError as e:
            with pytest.raises(spinf.SpinfError) as ee:
                spinf.Plan(inputs, token_budget=budget)
            assert ee.value.status_name == e.status
            continue
        _compare(spinf, inputs, token_budget=budget)


@pytest.mark.parametrize("bad", [
    [([1], [([], [[1]])])],
    [([1], [([1], [])])],
    [([1], [([1], [[]])])],
    [([1], [([1], [[2], [2]])])],
    [([], [])],
    [([1] * 4097, [([1], [[2]])])],
    [([1], [([1] * 257, [[2]])])],
    [([1], [([1], [[i] for i in range(1001)])])],
    [([1], [([1], [[2] * 6])])],
    [([1], [([1], [[2000]])])],
    [([1], [([1], None, -2)])],
    [([1], [([], None, 0)])],
    [([1], [([2000], None, 0)])],
])
def test_error_statuses_match(spinf, bad):
    with pytest.raises(op.PlanError) as e:
        op.plan(bad, vocab=1024)
    with pytest.raises(spinf.SpinfError) as ee:
        spinf.Plan(bad, vocab=1024)
    assert ee.value.status_name == e.value.status


def test_split_error_status(spinf):
    bad = [([1] * 8, [([1, 2, 3], [[1]])])]
    with pytest.raises(spinf.SpinfError) as ee:
        spinf.Plan(bad, token_budget=10)
    assert ee.value.status_name == "LIMIT"


def test_empty_request(spinf):
    Q = spinf.Plan([])
    assert Q.num_passes == 0 and Q.counts() == (0, 0)
    assert Q.collect([])["option_lp"].shape == (0,)


def test_collect_matches_oracle_collect(spinf):
    inputs = wl.stress(n_questions=50, content_tokens=100, vocab=1000)
    inputs = inputs + wl.tiny(vocab=1000)
    P, Q = _compare(spinf, inputs, token_budget=600)
    g = np.random.default_rng(3)
    tlps = [(-g.random(len(lay.gather_tok)) * 5).astype(np.float32) for lay in P.passes]
    ours = Q.collect(tlps)
    ref = oc.collect(P, tlps)
    flat = {k: [] for k in ("lp", "p", "floor_lp", "floor_p")}
    res, fres = [], []
    for per_q in ref:
        for r in per_q:
            for k in flat:
                flat[k].extend(r[k])
            res.append(r["residual"])
            fres.append(r["floor_residual"])
    np.testing.assert_allclose(ours["option_lp"], flat["lp"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ours["option_p"], flat["p"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ours["option_floor_lp"], flat["floor_lp"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ours["option_floor_p"], flat["floor_p"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ours["residual"], res, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ours["floor_residual"], fres, rtol=0, atol=1e-12)


def test_request_object_plans_identically(spinf):
    inputs = wl.stress(n_questions=30, content_tokens=120, vocab=1000) + wl.tiny(vocab=1000)
    req = spinf.Request(inputs)
    a, b = spinf.Plan(inputs, token_budget=700), spinf.Plan(req, token_budget=700)
    c = spinf.Plan(req, token_budget=700)
    assert a.num_passes == b.num_passes == c.num_passes
    for p in range(a.num_passes):
        ia, ib, ic = a.pass_info(p), b.pass_info(p), c.pass_info(p)
        for f in FIELDS:
            assert np.array_equal(getattr(ia, f), getattr(ib, f))
            assert np.array_equal(getattr(ia, f), getattr(ic, f))


def test_row_runs_deep_tries(spinf):
    """Option tries whose nodes are non-first children at every level: rows whose root
    path has more than four runs are flagged, every other row's runs are exact."""
    opts = [[1, 2, 5, 5, 5], [1, 3, 2, 5, 5], [1, 3, 3, 2, 5], [1, 3, 3, 3, 2]]
    inputs = [([7, 8, 9], [([4, 4], opts), ([6], opts)]), ([], [([2, 3], opts)])]
    P, Q = _compare(spinf, inputs)
    runs = Q.pass_info(0).row_runs
    assert (runs[:, 0] == -1).any() and (runs[:, 0] >= 0).any()


def test_row_runs_masks_match_visibility(spinf):
    """The attention kernel's run mask (a row's runs intersected with a scheduled KV tile's
    own keys, 64 columns at a time) equals k <= q < end[k] for every row of every tile."""
    inputs = wl.stress(n_questions=24, content_tokens=300, vocab=1000) + wl.tiny(vocab=1000)
    plan = spinf.Plan(inputs, token_budget=1024, vocab=1000)
    for p in range(plan.num_passes):
        info = plan.pass_info(p)
        for qt in range(info.n_qtiles):
            q = np.arange(qt * 128, qt * 128 + 128)
            real = q < info.T
            runs = info.row_runs[q].astype(np.int64)
            for e in range(int(info.tile_ptr[qt]), int(info.tile_ptr[qt + 1])):
                kv0, ln = int(info.tile_kv[e]), int(info.tile_len[e])
                keys = kv0 + np.arange(128)
                truth = (np.arange(128)[None, :] < ln) & (keys[None, :] <= q[:, None]) & \
                    (q[:, None] < info.end[np.minimum(keys, info.T_pad - 1)][None, :]) & real[:, None]
                got = np.zeros_like(truth)
                for i in range(4):
                    lo, hi = runs[:, 2 * i:2 * i + 1], runs[:, 2 * i + 1:2 * i + 2]
                    got |= (keys[None, :] >= lo) & (keys[None, :] < hi)
                got &= (np.arange(128)[None, :] < ln) & real[:, None]
                use = runs[:, 0] >= 0
                assert np.array_equal(got[use], truth[use]), (p, qt, e)


@pytest.mark.parametrize("window", [1, 7, 64, 200, 100000])
def test_window_schedule_is_exact(spinf, window):
    """A tile stays in the windowed schedule iff some row of its Q tile sees some key of
    it within the window (oracle visible sets and depths, brute force)."""
    inputs = wl.stress(n_questions=24, content_tokens=300, vocab=1000) + wl.tiny(vocab=1000)
    P = op.plan(inputs, token_budget=1024, vocab=1000)
    plan = spinf.Plan(inputs, token_budget=1024, vocab=1000)
    for p, lay in enumerate(P.passes):
        tp, tk, tl = plan.window_schedule(p, window)
        want_ptr, want_kv = [0], []
        for qt in range(lay.T_pad // 128):
            rows = range(qt * 128, min(qt * 128 + 128, lay.T))
            vis = {q: set(lay.visible(q)) for q in rows}
            for e in range(lay.tile_ptr[qt], lay.tile_ptr[qt + 1]):
                kv0, ln = int(lay.tile_kv[e]), int(lay.tile_len[e])
                if any(k in vis[q] and lay.pos[q] - lay.pos[k] < window for q in rows for k in range(kv0, kv0 + ln)):
                    want_kv.append((kv0, ln))
            want_ptr.append(len(want_kv))
        assert tp.tolist() == want_ptr
        assert list(zip(tk.tolist(), tl.tolist())) == want_kv
        if window >= 100000:   # a window that never bites keeps every tile
            assert np.array_equal(tk, lay.tile_kv) and np.array_equal(tl, lay.tile_len)


@pytest.mark.parametrize("window,key_tile", [(0, 128), (0, 64), (7, 64), (64, 64), (200, 64)])
def test_tile_schedule_is_exact(spinf, window, key_tile):
    """The schedule the attention kernel runs (64-key tiles at d_head 256): each planner
    tile taken whole or as its two 64-key halves, a piece kept iff some row of its Q tile
    sees one of its keys (within the window), in the planner's order (oracle visible sets
    and depths, brute force).  Window 0 with 128-key tiles is the planner's own schedule."""
    inputs = wl.stress(n_questions=24, content_tokens=300, vocab=1000) + wl.tiny(vocab=1000)
    P = op.plan(inputs, token_budget=1024, vocab=1000)
    plan = spinf.Plan(inputs, token_budget=1024, vocab=1000)
    n_halves_dropped = 0
    for p, lay in enumerate(P.passes):
        tp, tk, tl = plan.tile_schedule(p, window, key_tile)
        want_ptr, want_kv = [0], []
        for qt in range(lay.T_pad // 128):
            rows = range(qt * 128, min(qt * 128 + 128, lay.T))
            vis = {q: set(lay.visible(q)) for q in rows}
            for e in range(lay.tile_ptr[qt], lay.tile_ptr[qt + 1]):
                kv0, ln = int(lay.tile_kv[e]), int(lay.tile_len[e])
                for sub in range(0, 128, key_tile):
                    n = min(ln - sub, key_tile)
                    if n <= 0:
                        break
                    keys = range(kv0 + sub, kv0 + sub + n)
                    if any(k in vis[q] and (window == 0 or lay.pos[q] - lay.pos[k] < window)
                           for q in rows for k in keys):
                        want_kv.append((kv0 + sub, n))
                    else:
                        n_halves_dropped += 1
            want_ptr.append(len(want_kv))
        assert tp.tolist() == want_ptr, p
        assert list(zip(tk.tolist(), tl.tolist())) == want_kv, p
        if (window, key_tile) == (0, 128):
            assert np.array_equal(tk, lay.tile_kv) and np.array_equal(tl, lay.tile_len)
    if (window, key_tile) == (0, 128):
        assert n_halves_dropped == 0          # the planner schedules no tile that no row sees
    else:
        assert n_halves_dropped > 0           # the case does exercise the dropping


def test_tile_schedule_rejects_bad_arguments(spinf):
    plan = spinf.Plan(wl.tiny(vocab=1000), vocab=1000)
    for args in ((0, -1, 64), (0, 0, 32), (0, 0, 256), (5, 0, 64)):
        with pytest.raises(spinf.SpinfError) as e:
            plan.tile_schedule(*args)
        assert e.value.status_name == "INVALID"


def _searched_request(g, n_inputs, vocab=60):
    """Inputs mixing scored questions and searched slots (token sets -1..3)."""
    inputs = []
    for _ in range(n_inputs):
        content = g.integers(0, vocab, size=int(g.integers(0, 200))).tolist()
        qs = []
        for _ in range(int(g.integers(0 if content else 1, 7))):
            template = g.integers(0, vocab, size=int(g.integers(1, 15))).tolist()
            if g.random() < 0.4:
                qs.append((template, None, int(g.integers(-1, 4))))
                continue
            opts, seen = [], set()
            for _ in range(int(g.integers(1, 4))):
                o = tuple(g.integers(0, 6, size=int(g.integers(1, 3))).tolist())
                if o not in seen:
                    seen.add(o)
                    opts.append(list(o))
            qs.append((template, opts))
        if not content and not qs:
            content = [1]
        inputs.append((content, qs))
    return inputs


@pytest.mark.parametrize("budget", [128, 400, 16384])
def test_searched_slots_bit_exact(spinf, budget):
    g = np.random.default_rng(budget)
    for trial in range(12):
        inputs = _searched_request(g, int(g.integers(1, 10)))
        k = int(g.integers(1, 17))
        try:
            op.plan(inputs, token_budget=budget, extract_k=k)
        except op.PlanError as e:
            with pytest.raises(spinf.SpinfError) as ee:
                spinf.Plan(inputs, token_budget=budget, extract_k=k)
            assert ee.value.status_name == e.status
            continue
        P, Q = _compare(spinf, inputs, token_budget=budget, extract_k=k)
        n_x = sum(sum(row) for row in P.searched)
        assert Q.extract_counts() == (n_x, k)
        assert Q.counts()[0] == sum(P.n_questions)


@pytest.mark.parametrize("k", [0, 17])
def test_extract_k_range(spinf, k):
    with pytest.raises(op.PlanError):
        op.plan([([1], [([2], None, -1)])], extract_k=k)
    with pytest.raises(spinf.SpinfError) as ee:
        spinf.Plan([([1], [([2], None, -1)])], extract_k=k)
    assert ee.value.status_name == "INVALID"


def test_collect_extract_matches_oracle(spinf):
    g = np.random.default_rng(11)
    inputs = _searched_request(g, 9)
    P, Q = _compare(spinf, inputs, token_budget=300, extract_k=5)
    toks = [g.integers(-1, 60, size=(len(lay.x_m), 5)).astype(np.int32) for lay in P.passes]
    lps = [(-g.random((len(lay.x_m), 5)) * 9).astype(np.float32) for lay in P.passes]
    tok, lp = Q.collect_extract(toks, lps)
    ref = oc.collect_extract(P, toks, lps)
    assert tok.shape == (len(ref), 5)
    for i, (t, l) in enumerate(ref):
        assert tok[i].tolist() == t.tolist()
        np.testing.assert_array_equal(lp[i], l)
    tlps = [(-g.random(len(lay.gather_tok)) * 5).astype(np.float32) for lay in P.passes]
    ours = Q.collect(tlps)
    flat_res = [np.nan if r is None else r["residual"] for per_q in oc.collect(P, tlps) for r in per_q]
    np.testing.assert_allclose(ours["residual"], flat_res, rtol=0, atol=1e-12)


def _grid(g, vocab=60):
    n_ph = int(g.integers(0, 4))
    segments = [g.integers(0, vocab, size=int(g.integers(0, 5))).tolist() for _ in range(n_ph + 1)]
    if not any(segments):
        segments[-1] = [int(g.integers(0, vocab))]
    values = [[g.integers(0, vocab, size=int(g.integers(0, 3))).tolist() for _ in range(int(g.integers(1, 4)))]
              for _ in range(n_ph)]
    if g.random() < 0.3:
        return (segments, values, None, int(g.integers(-1, 2)))
    opts = [[int(x)] for x in g.choice(vocab, size=int(g.integers(1, 4)), replace=False)]
    return (segments, values, opts)


@pytest.mark.parametrize("budget", [200, 16384])
def test_grids_bit_exact(spinf, budget):
    g = np.random.default_rng(budget + 1)
    for trial in range(12):
        inputs = []
        for c, qs in _searched_request(g, int(g.integers(1, 6))):
            inputs.append((c, qs, [_grid(g) for _ in range(int(g.integers(0, 3)))]))
        try:
            op.plan(inputs, token_budget=budget)
        except op.PlanError as e:
            with pytest.raises(spinf.SpinfError) as ee:
                spinf.Plan(inputs, token_budget=budget)
            assert ee.value.status_name == e.status
            continue
        P, Q = _compare(spinf, inputs, token_budget=budget)
        assert Q.counts()[0] == sum(P.n_questions)


@pytest.mark.parametrize("bad,status", [
    ([([1], [], [([[1], [2]], [[]], [[3]])])], "INVALID"),
    ([([1], [], [([[1], [2], [4]], [[[5], [6]], [[7], [8], [9]]], [[3]])])], "LIMIT"),
    ([([1], [], [([[]], [], [[3]])])], "INVALID"),
])
def test_grid_error_statuses_match(spinf, bad, status):
    with pytest.raises(op.PlanError) as e:
        op.plan(bad, max_prompts_per_input=5)
    with pytest.raises(spinf.SpinfError) as ee:
        spinf.Plan(bad, max_prompts_per_input=5)
    assert e.value.status == ee.value.status_name == status


@pytest.mark.parametrize("name", ["tiny", "wikinews", "moderation"])
@pytest.mark.parametrize("window", [0, 9])
def test_derived_schedules_are_exact(spinf, name, window):
    """The schedules the attention kernel runs (64-key tiles; 64-row Q tiles) against brute
    force: a KV tile is listed for a Q tile iff some row of the Q tile sees one of its keys
    (within the window); a 64-row Q tile of pad rows only lists one tile (masked for all its
    rows, so that the kernel writes its pad rows).  Tiles appear in the planner's order."""
    f, shape = wl.WORKLOADS[name]
    inputs = f()
    P = op.plan(inputs, vocab=shape.vocab)
    Q = spinf.Plan(inputs, vocab=shape.vocab)
    for p, lay in enumerate(P.passes[:2]):
        end, pos = lay.end, lay.pos
        for key_tile, q_rows in ((64, 128), (64, 64), (128, 64)):
            tp, tk, tl = Q.tile_schedule(p, window, key_tile, q_rows)
            assert len(tp) == lay.T_pad // q_rows + 1
            for qt in range(lay.T_pad // q_rows):
                r0, r1 = qt * q_rows, min((qt + 1) * q_rows, lay.T)
                want = []
                qp = qt * q_rows // 128
                for e in range(lay.tile_ptr[qp], lay.tile_ptr[qp + 1]):
                    for sub in range(0, 128, key_tile):
                        kv0, n = int(lay.tile_kv[e]) + sub, min(int(lay.tile_len[e]) - sub, key_tile)
                        if n <= 0:
                            break
                        if any(max(k, r0) < min(int(end[k]), r1) and
                               (window <= 0 or min(int(pos[q]) for q in range(max(k, r0), min(int(end[k]), r1)))
                                - int(pos[k]) < window) for k in range(kv0, kv0 + n)):
                            want.append((kv0, n))
                got = list(zip(tk[tp[qt]:tp[qt + 1]].tolist(), tl[tp[qt]:tp[qt + 1]].tolist()))
                if r1 <= r0:   # pad rows only
                    assert len(got) == 1, (qt, got)
                else:
                    assert got == want, (name, p, key_tile, q_rows, qt)
