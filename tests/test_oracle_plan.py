"""Pins of the oracle planner: hand-derived layouts and the root-path invariant.

The expected arrays below were worked out by hand from the layout rules
(content first, then each question's template, then its option-trie nodes in
pre-order; a branch sees its own content and its own root path only), not by
running any planner.
"""
import numpy as np
import pytest

from oracle import plan as op
from synth import workloads as wl

PAD = -1


def _check_pads(lay):
    for r in range(lay.T, lay.T_pad):
        assert lay.tok[r] == 0 and lay.parent[r] == -1 and lay.pos[r] == 0
        assert lay.end[r] == r + 1 and lay.anchor[r] == r


def test_single_question_with_floor():
    P = op.plan([([10, 11, 12], [([20, 21], [[30], [31]])])])
    assert len(P.passes) == 1
    L = P.passes[0]
    assert L.T == 7 and L.T_pad == 128
    assert L.tok[:7].tolist() == [10, 11, 12, 20, 21, 20, 21]
    assert L.parent[:7].tolist() == [-1, 0, 1, 2, 3, -1, 5]
    assert L.pos[:7].tolist() == [0, 1, 2, 3, 4, 0, 1]
    assert L.end[:7].tolist() == [5, 5, 5, 5, 5, 7, 7]
    assert L.anchor[:7].tolist() == [0, 0, 0, 0, 0, 5, 5]
    assert L.slot_row.tolist() == [4, 6]
    assert L.gather_m.tolist() == [0, 0, 1, 1]
    assert L.gather_tok.tolist() == [30, 31, 30, 31]
    assert L.tile_ptr.tolist() == [0, 2]
    assert L.tile_kv.tolist() == [0, 5]
    assert L.tile_len.tolist() == [5, 2]
    _check_pads(L)


def test_sibling_branches_do_not_see_each_other():
    P = op.plan([([1, 2], [([3], [[4], [5]]), ([6, 7], [[8]])])], floors=False)
    L = P.passes[0]
    assert L.tok[:5].tolist() == [1, 2, 3, 6, 7]
    assert L.parent[:5].tolist() == [-1, 0, 1, 1, 3]
    assert L.pos[:5].tolist() == [0, 1, 2, 2, 3]
    assert L.end[:5].tolist() == [5, 5, 3, 5, 5]
    assert L.visible(3) == [0, 1, 3]
    assert L.visible(4) == [0, 1, 3, 4]
    assert L.slot_row.tolist() == [2, 4]
    assert L.gather_m.tolist() == [0, 0, 1]
    assert L.gather_tok.tolist() == [4, 5, 8]


def test_option_trie_rows():
    P = op.plan([([1], [([2], [[5, 6], [5, 7], [8]])])], floors=False)
    L = P.passes[0]
    assert L.tok[:3].tolist() == [1, 2, 5]
    assert L.parent[:3].tolist() == [-1, 0, 1]
    assert L.pos[:3].tolist() == [0, 1, 2]
    assert L.end[:3].tolist() == [3, 3, 3]
    assert L.slot_row.tolist() == [1, 2]
    assert L.gather_m.tolist() == [0, 1, 0, 1, 0]
    assert L.gather_tok.tolist() == [5, 6, 5, 7, 8]


def test_trie_preorder_and_first_insertion():
    assert op.trie_nodes([[5, 6, 7], [9, 1], [5, 8]]) == [(5,), (5, 6), (9,)]
    # first insertion, not token order: 9 was inserted before 5
    assert op.trie_nodes([[9, 1], [5, 6, 7], [5, 8], [9, 3, 4]]) == [(9,), (9, 3), (5,), (5, 6)]
    P = op.plan([([], [([2, 3], [[5, 6, 7], [9, 1], [5, 8]])])], floors=False)
    L = P.passes[0]
    # rows: 0:2 1:3(slot) 2:(5,) 3:(5,6) 4:(9,)
    assert L.tok[:5].tolist() == [2, 3, 5, 6, 9]
    assert L.parent[:5].tolist() == [-1, 0, 1, 2, 1]
    assert L.pos[:5].tolist() == [0, 1, 2, 3, 2]
    assert L.end[:5].tolist() == [5, 5, 4, 4, 5]
    assert L.slot_row.tolist() == [1, 2, 3, 4]
    # option [5,6,7]: rows 1,2,3; [9,1]: rows 1,4; [5,8]: rows 1,2
    assert L.gather_m.tolist() == [0, 1, 2, 0, 3, 0, 1]
    assert L.gather_tok.tolist() == [5, 6, 7, 9, 1, 5, 8]


def test_next_fit_and_split():
    # budget 10: input0 = 4 + 2 = 6; input1 = 3 + 2 = 5 -> new pass; floors (sizes 2, 2)
    inputs = [([1, 2, 3, 4], [([5, 6], [[7]])]), ([1, 2, 3], [([8, 9], [[7]])])]
    P = op.plan(inputs, token_budget=10)
    assert [p.T for p in P.passes] == [6, 9]
    # an input that brings the pass to exactly the budget stays in it (a pass holds <= budget rows)
    P = op.plan(inputs, token_budget=11, floors=False)
    assert [p.T for p in P.passes] == [11]
    # long input split: content 4 + questions of 3 each, budget 10 -> chunks of 2 questions
    inputs = [([1, 2, 3, 4], [([5, 6, 7], [[1]]), ([5, 6, 8], [[1]]), ([5, 6, 9], [[1]])])]
    P = op.plan(inputs, token_budget=10, floors=False)
    assert [p.T for p in P.passes] == [10, 7]
    assert [u.qidx for p in P.passes for u in p.units] == [[0, 1], [2]]
    assert P.passes[1].tok[:7].tolist() == [1, 2, 3, 4, 5, 6, 9]


def test_floors_dedup_in_first_appearance_order():
    q1 = ([5, 6], [[7], [8]])
    q2 = ([9], [[7], [8]])
    P = op.plan([([1], [q1, q2]), ([2], [q2, q1])])
    L = P.passes[0]
    floors = [u for u in L.units if u.source < 0]
    assert [u.questions[0][0] for u in floors] == [(5, 6), (9,)]
    P2 = op.plan([([1], [q1, q2])], floor_prefix=[3, 4])
    fl = [u for u in P2.passes[0].units if u.source < 0]
    assert all(u.content == (3, 4) for u in fl)


@pytest.mark.parametrize("bad,status", [
    ([([1], [([], [[1]])])], "INVALID"),
    ([([1], [([1], [])])], "INVALID"),
    ([([1], [([1], [[]])])], "INVALID"),
    ([([1], [([1], [[2], [2]])])], "INVALID"),
    ([([], [])], "INVALID"),
    ([([1] * 4097, [([1], [[2]])])], "LIMIT"),
    ([([1], [([1] * 257, [[2]])])], "LIMIT"),
    ([([1], [([1], [[2]] * 0 + [[i] for i in range(1001)])])], "LIMIT"),
    ([([1], [([1], [[2] * 6])])], "LIMIT"),
    ([([1], [([1], [[2000]])])], "INVALID"),
])
def test_errors(bad, status):
    with pytest.raises(op.PlanError) as e:
        op.plan(bad, vocab=1024)
    assert e.value.status == status


def _at_limits():
    """One input at each of the man page's limits (PARAMETERS): content 4096 tokens, template
    256, 1000 options, an option of 5 tokens."""
    return [([1] * 4096, [([2], [[3]])]),
            ([1], [([2] * 256, [[3]])]),
            ([1], [([2], [[t] for t in range(1000)])]),
            ([1], [([2], [[3, 4, 5, 6, 7], [3]])])]


def test_limits_are_inclusive():
    """An input exactly at a limit is accepted; one token or option more is refused."""
    for inp in _at_limits():
        op.plan([inp])
    over = [([1] * 4097, [([2], [[3]])]), ([1], [([2] * 257, [[3]])]),
            ([1], [([2], [[t] for t in range(1001)])]), ([1], [([2], [[3, 4, 5, 6, 7, 8], [3]])])]
    for inp in over:
        with pytest.raises(op.PlanError) as e:
            op.plan([inp])
        assert e.value.status == "LIMIT"


def test_floor_exactly_at_the_budget():
    """A question of 10 rows (9 template tokens, one 2-token option: one trie node) at budget 10:
    its floor is exactly 10 rows and fits; with a one-token floor prefix it does not."""
    inputs = [([], [([2] * 9, [[3, 4]])])]
    P = op.plan(inputs, token_budget=10)
    assert [p.T for p in P.passes] == [10, 10]
    with pytest.raises(op.PlanError) as e:
        op.plan(inputs, token_budget=10, floor_prefix=[7])
    assert e.value.status == "LIMIT"


def test_split_error_when_question_does_not_fit():
    with pytest.raises(op.PlanError) as e:
        op.plan([([1] * 8, [([1, 2, 3], [[1]])])], token_budget=10)
    assert e.value.status == "LIMIT"


def _logical_checks(inputs, P):
    """Every row sees exactly its logical root path, read off the input description."""
    for lay in P.passes:
        tok = lay.tok
        for u in lay.units:
            s, L = u.start, len(u.content)
            for i in range(L):
                assert [int(tok[k]) for k in lay.visible(s + i)] == list(u.content[: i + 1])
        for rec in lay.questions:
            if rec.source >= 0:
                unit = next(u for u in lay.units if u.source == rec.source and rec.qidx in u.qidx)
                template, options = inputs[rec.source][1][rec.qidx]
            else:
                unit = next(u for u in lay.units if u.source < 0 and u.floor_key == rec.key)
                template, options = rec.key
            content = list(unit.content)
            for o, gs in zip(options, rec.option_gather):
                for i, g in enumerate(gs):
                    row = int(lay.slot_row[lay.gather_m[g]])
                    want = content + list(template) + list(o[:i])
                    assert [int(tok[k]) for k in lay.visible(row)] == want
                    assert lay.pos[row] == len(want) - 1
                    assert lay.gather_tok[g] == o[i]
        # end[] agrees with the visible sets: row q sees k iff k <= q < end[k]
        T = lay.T
        for q in range(0, T, max(1, T // 257)):
            vis = set(lay.visible(q))
            lo = int(lay.anchor[q])
            hi = max(k for k in range(lo, T) if lay.anchor[k] == lo) + 1
            for k in range(lo, hi):
                assert (k in vis) == (k <= q < lay.end[k])


@pytest.mark.parametrize("name", ["tiny", "wikinews", "stress"])
def test_root_path_invariant(name):
    f, shape = wl.WORKLOADS[name]
    inputs = f()
    P = op.plan(inputs, vocab=shape.vocab)
    _logical_checks(inputs, P)


def test_root_path_invariant_small_budget_trie():
    inputs = wl.stress(n_questions=40, content_tokens=300)
    P = op.plan(inputs, token_budget=1024, vocab=151936)
    assert len(P.passes) > 1
    _logical_checks(inputs, P)


def test_schedule_is_exact():
    """A KV tile is scheduled iff some row of the Q tile sees some key in it."""
    inputs = wl.stress(n_questions=30, content_tokens=700)
    P = op.plan(inputs, token_budget=2048, vocab=151936)
    for lay in P.passes:
        sched = {}
        for qt in range(lay.T_pad // 128):
            sched[qt] = lay.tile_kv[lay.tile_ptr[qt]:lay.tile_ptr[qt + 1]].tolist()
        for qt in range(lay.T_pad // 128):
            want = []
            for u in lay.units:
                s, e = u.start, u.start + u.size
                rows = range(max(qt * 128, s), min(qt * 128 + 128, e))
                if not len(rows):
                    continue
                js = sorted({(k - s) // 128 for q in rows for k in lay.visible(q)})
                want += [s + 128 * j for j in js]
                for j in js:   # every key a row of this unit sees lies inside its unit
                    assert lay.tile_len[list(lay.tile_kv).index(s + 128 * j)] == min(128, e - s - 128 * j)
            assert sched[qt] == want


def test_packing_order_does_not_change_an_inputs_layout():
    inputs = wl.tiny()
    a = op.plan(inputs, floors=False)
    b = op.plan(inputs[::-1], floors=False)
    la, lb = a.passes[0], b.passes[0]
    ua = la.units[0]
    ub = next(u for u in lb.units if u.source == 1)
    n = ua.size
    for arr in ("tok", "pos"):
        assert np.array_equal(getattr(la, arr)[ua.start:ua.start + n], getattr(lb, arr)[ub.start:ub.start + n])
    assert np.array_equal(la.end[:n] - ua.start, lb.end[ub.start:ub.start + n] - ub.start)
