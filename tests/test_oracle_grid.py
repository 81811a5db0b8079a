"""Pins of the oracle's placeholder grids: hand-expanded cells and the layout of a grid
equal to that of the same questions written out by hand."""
import pytest

from oracle import plan as op

GRID = ([[1, 2], [3], [4]], [[[10], [11, 12]], [[20], [21], [22]]], [[30], [31]])


def test_cells_by_hand():
    cells = op.expand_grid(GRID)
    assert [c[0] for c in cells] == [
        [1, 2, 10, 3, 20, 4], [1, 2, 10, 3, 21, 4], [1, 2, 10, 3, 22, 4],
        [1, 2, 11, 12, 3, 20, 4], [1, 2, 11, 12, 3, 21, 4], [1, 2, 11, 12, 3, 22, 4]]
    assert all(c[1] == [[30], [31]] for c in cells)
    assert op.grid_size(GRID) == 6


def test_searched_grid_and_empty_pieces():
    grid = ([[], [5]], [[[7], [], [8, 9]]], None, 2)
    assert op.expand_grid(grid) == [([7, 5], None, 2), ([5], None, 2), ([8, 9, 5], None, 2)]


def test_grid_plans_like_its_written_out_questions():
    own = [([50], [[60], [61]])]
    by_hand = [(c[0], c[1]) for c in op.expand_grid(GRID)]
    P = op.plan([([9, 9, 9], own, [GRID])])
    Q = op.plan([([9, 9, 9], own + by_hand)])
    assert P.n_questions == Q.n_questions == [7]
    for a, b in zip(P.passes, Q.passes):
        for f in ("tok", "parent", "pos", "end", "tile_kv", "slot_row", "gather_m", "gather_tok"):
            assert getattr(a, f).tolist() == getattr(b, f).tolist(), f
    assert P.question_home == Q.question_home and set(P.floor_home) == set(Q.floor_home)


def test_grid_errors():
    with pytest.raises(op.PlanError) as e:
        op.plan([([1], [], [([[1], [2]], [], [[3]])])])            # two segments, no placeholder
    assert e.value.status == "INVALID"
    with pytest.raises(op.PlanError) as e:
        op.plan([([1], [], [([[1], [2]], [[]], [[3]])])])          # a placeholder without values
    assert e.value.status == "INVALID"
    with pytest.raises(op.PlanError) as e:
        op.plan([([1], [], [GRID])], max_prompts_per_input=5)      # 6 cells
    assert e.value.status == "LIMIT"
    with pytest.raises(op.PlanError) as e:
        op.plan([([1], [], [([[]], [], [[3]])])])                  # a cell with an empty template
    assert e.value.status == "INVALID"


def test_synthetic_written_out_form_matches_the_expansion():
    """synth's written-out form of a grid request (the bench's comparison input) has the cells
    in the plan's order: the same layout as the grid request itself."""
    from synth import workloads as wl

    searched = ([[], [5]], [[[7], [], [8, 9]]], None, 2)
    inputs = [([9, 9, 9], [([50], [[60], [61]])], [GRID, searched])] + wl.wikinews_grid(vocab=1000, n_contents=3)
    written = wl.written_out(inputs)
    assert written[0][1][1:] == [tuple(c) for c in op.expand_grid(GRID)] + op.expand_grid(searched)
    P, Q = op.plan(inputs, vocab=1000), op.plan(written, vocab=1000)
    assert len(P.passes) == len(Q.passes)
    for a, b in zip(P.passes, Q.passes):
        for f in ("tok", "parent", "pos", "end", "slot_row", "gather_tok"):
            assert getattr(a, f).tolist() == getattr(b, f).tolist(), f
