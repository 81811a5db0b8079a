"""Oracle pack planner (integer work; TEST INFRASTRUCTURE ONLY, see ``oracle/__init__``).

What it restates, page by page:

* "spinf-serve 0.1.1" (PyPI), "What it does": a question is a template that
  ends where the answer goes, with the answers to score there; the content is
  read once and every question is a branch of the same pass; each question
  also gets a floor, the same question on empty content.
* same page, "Speed and scale": contents and their question branches are
  packed into 16k-token passes; a branch sees its own content, never a
  sibling branch or another packed input.
* same page, "Layout": templates become token tries (the options of one
  question share their common prefixes).
* "spinf-serve" man page, PARAMETERS: ``--token-budget`` 16384 tokens per pass,
  ``--max-content-tokens`` 4096, ``--max-query-tokens`` 256,
  ``--max-prompts-per-input`` 10000, ``--max-options`` 1000,
  ``--max-option-tokens`` 5, ``--max-tokens`` (largest single input).
* same page, CAVEATS: long inputs run alone.
* same page, "What it does": placeholders turn one template into a grid of
  questions.
* "spinf-serve 0.1.1" (PyPI), "What it does" and the man page's DESCRIPTION:
  extraction slots (``{*}`` text, ``{n}`` numbers, ``{$}`` amounts) ride the
  same read; the engine returns the most likely answers with their
  probabilities.

Readings where the pages are silent (each is listed in the design notes):

1. The slot is the last template token: the next-token distribution there
   scores the first option token.
2. A multi-token option is scored by the sum of its token log-probabilities;
   only proper prefixes of options are laid out (trie nodes), in pre-order,
   children in order of first insertion.
3. One floor input per distinct (template, options) pair, in order of first
   appearance, after all user inputs; its content is ``floor_prefix``
   (empty by default).
4. Packing is next-fit in submission order.  An input larger than the budget
   is split into chunks, each the full content plus a greedy run of the
   remaining questions; it is an error when the content and the next question
   do not fit together.
5. Position ids are tree depth (length of the root path minus one).
6. The pass is padded to a multiple of 128 rows; a pad row sees nothing and
   its output is unspecified.
7. A searched slot (``{*}``, ``{n}``, ``{$}``) is a template with no options:
   its template rows are laid out like a scored question's, its last template
   row is a scoring row, and the ``extract_k`` most likely next tokens there,
   among an allowed-token set named by the question (``-1``: every token), are
   returned with their log-probabilities.  Later decoding steps append the
   chosen tokens to the template and plan again.  A searched slot gets no
   floor (the pages give the floor for scored questions only).

8. A grid is a template written as literal segments around placeholders, each
   placeholder with a list of values (token sequences).  It stands for one
   question per combination of values, the first placeholder varying slowest;
   every cell is an ordinary question with the grid's options (or a searched
   slot).  An input's grid cells follow its own questions, grid by grid, and
   count toward ``max_prompts_per_input``.

A question is ``(template, options)`` (scored) or ``(template, None, token_set)``
(a searched slot).  A grid is ``(segments, values, options)`` or
``(segments, values, None, token_set)``.  An input is ``(content, questions)``
or ``(content, questions, grids)``.

The visible-key set of a row is kept in its plainest form: the content rows of
its own input up to itself (content rows) or all of them (branch rows), plus
the branch rows on its own root path.  Everything else (``end``, ``pos``, the
KV-tile schedule) is derived from that set by its definition.
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass, field

import numpy as np

TILE = 128

#: Defaults from the man page's PARAMETERS section.  ``max_tokens`` has no
#: stated default; it is read as the per-request processed-token limit.
DEFAULTS = {
    "token_budget": 16384,
    "max_tokens": 2_000_000,
    "max_content_tokens": 4096,
    "max_query_tokens": 256,
    "max_options": 1000,
    "max_option_tokens": 5,
    "max_prompts_per_input": 10000,
    "floors": True,
    "floor_prefix": (),
    "vocab": 0,
    "extract_k": 8,
}


def is_searched(question):
    """A searched slot is written ``(template, None, token_set)``."""
    return len(question) == 3 and question[1] is None


class PlanError(Exception):
    """A rejected request.  ``status`` is ``"INVALID"`` or ``"LIMIT"``."""

    def __init__(self, status: str, message: str):
        super().__init__(f"{status}: {message}")
        self.status = status


def trie_nodes(options):
    """Proper prefixes of the options laid out as trie nodes, in pre-order.

    A node is a prefix ``(t1..ti)``, ``i >= 1``, of an option longer than ``i``.
    Children are ordered by first insertion; options are inserted in the given
    order.
    """
    root: dict = {}
    for opt in options:
        node = root
        for t in opt[:-1]:
            node = node.setdefault(t, {})
    out = []

    def walk(node, prefix):
        for t, child in node.items():
            p = prefix + (t,)
            out.append(p)
            walk(child, p)

    walk(root, ())
    return out


def expand_grid(grid):
    """The questions of one grid, first placeholder slowest (reading 8)."""
    segments, values = grid[0], grid[1]
    cells = []
    for combo in itertools.product(*values):
        template = list(segments[0])
        for value, seg in zip(combo, segments[1:]):
            template += list(value) + list(seg)
        cells.append((template, None, grid[3]) if grid[2] is None else (template, grid[2]))
    return cells


def grid_size(grid):
    """Number of cells of a grid, without expanding it."""
    n = 1
    for v in grid[1]:
        n *= len(v)
    return n


def _expand_inputs(inputs, o):
    """Inputs with their grids expanded into trailing questions: ``(content, questions)``."""
    out = []
    for i, inp in enumerate(inputs):
        content, questions = inp[0], list(inp[1])
        grids = inp[2] if len(inp) > 2 else ()
        total = len(questions)
        for grid in grids:
            if len(grid[0]) != len(grid[1]) + 1:
                raise PlanError("INVALID", f"input {i}: a grid needs one more segment than placeholders")
            if any(len(v) == 0 for v in grid[1]):
                raise PlanError("INVALID", f"input {i}: a grid placeholder without values")
            total += grid_size(grid)
            if total > o["max_prompts_per_input"]:
                raise PlanError("LIMIT", f"input {i}: more questions than max_prompts_per_input")
        for grid in grids:
            questions += expand_grid(grid)
        out.append((content, questions))
    return out


def question_size(template, options):
    """Rows of one laid-out question: its template and its option-trie nodes
    (``options`` is None for a searched slot: the template only)."""
    return len(template) + (0 if options is None else len(trie_nodes(options)))


@dataclass
class Unit:
    """One laid-out input: a user input (or a chunk of one) or a floor."""

    source: int            # user input index, or -1 for a floor
    qidx: list             # question indices of the source input held here
    content: tuple
    questions: list        # [(template, options)]
    floor_key: object = None
    size: int = 0
    start: int = 0         # first packed row, set at layout


@dataclass
class QuestionRecord:
    """Where one laid-out question's scores live."""

    source: int            # user input index, or -1 for a floor
    qidx: int
    key: object            # (template, options) as tuples: the floor lookup key
    option_gather: list    # per option: list of gather indices, in token order
    extract: int = -1      # searched slot: its index in the pass's extraction list


@dataclass
class PassLayout:
    T: int
    T_pad: int
    tok: np.ndarray
    parent: np.ndarray
    pos: np.ndarray
    end: np.ndarray
    anchor: np.ndarray
    tile_ptr: np.ndarray
    tile_kv: np.ndarray
    tile_len: np.ndarray
    slot_row: np.ndarray
    gather_m: np.ndarray
    gather_tok: np.ndarray
    x_m: np.ndarray        # [X] scoring-row index of each searched slot, in layout order
    x_set: np.ndarray      # [X] its allowed-token set (-1: any token)
    units: list
    questions: list
    # visible-set representation, per real row (global rows)
    content_lo: np.ndarray = None
    content_hi: np.ndarray = None
    chain: list = field(default_factory=list)

    def visible(self, q):
        """Sorted global rows whose keys row ``q`` sees (its root path)."""
        lo, hi = int(self.content_lo[q]), int(self.content_hi[q])
        return list(range(lo, hi)) + list(self.chain[q])


@dataclass
class Plan:
    passes: list
    n_inputs: int
    n_questions: list      # per user input
    n_options: list        # per user input: list per question (0 for a searched slot)
    searched: list         # per user input: list per question of bools
    extract_k: int
    question_home: dict    # (input, qidx) -> (pass, record index)
    floor_home: dict       # floor key -> (pass, record index)


def _key(template, options):
    return (tuple(template), tuple(tuple(o) for o in options))


def _validate(inputs, o):
    vocab = o["vocab"]
    if not (1 <= o["extract_k"] <= 16):
        raise PlanError("INVALID", "extract_k must be in 1..16")

    def ids_ok(ids):
        return vocab <= 0 or all(0 <= t < vocab for t in ids)

    if not ids_ok(o["floor_prefix"]):
        raise PlanError("INVALID", "floor prefix token out of range")
    for i, (content, questions) in enumerate(inputs):
        if len(content) > o["max_content_tokens"]:
            raise PlanError("LIMIT", f"input {i}: content longer than max_content_tokens")
        if len(questions) > o["max_prompts_per_input"]:
            raise PlanError("LIMIT", f"input {i}: more questions than max_prompts_per_input")
        if not ids_ok(content):
            raise PlanError("INVALID", f"input {i}: content token out of range")
        if len(content) == 0 and len(questions) == 0:
            raise PlanError("INVALID", f"input {i}: nothing to read")
        size = len(content)
        for j, question in enumerate(questions):
            template, options = question[0], question[1]
            if len(template) == 0:
                raise PlanError("INVALID", f"input {i} question {j}: empty template")
            if len(template) > o["max_query_tokens"]:
                raise PlanError("LIMIT", f"input {i} question {j}: template longer than max_query_tokens")
            if is_searched(question):
                if not isinstance(question[2], int) or question[2] < -1:
                    raise PlanError("INVALID", f"input {i} question {j}: bad token set")
                if not ids_ok(template):
                    raise PlanError("INVALID", f"input {i} question {j}: template token out of range")
                size += len(template)
                continue
            if options is None or len(options) == 0:
                raise PlanError("INVALID", f"input {i} question {j}: no options")
            if len(options) > o["max_options"]:
                raise PlanError("LIMIT", f"input {i} question {j}: more options than max_options")
            seen = set()
            for opt in options:
                if len(opt) == 0:
                    raise PlanError("INVALID", f"input {i} question {j}: empty option")
                if len(opt) > o["max_option_tokens"]:
                    raise PlanError("LIMIT", f"input {i} question {j}: option longer than max_option_tokens")
                if tuple(opt) in seen:
                    raise PlanError("INVALID", f"input {i} question {j}: duplicate option")
                seen.add(tuple(opt))
                if not ids_ok(opt):
                    raise PlanError("INVALID", f"input {i} question {j}: option token out of range")
            if not ids_ok(template):
                raise PlanError("INVALID", f"input {i} question {j}: template token out of range")
            size += question_size(template, options)
        if size > o["max_tokens"]:
            raise PlanError("LIMIT", f"input {i}: larger than max_tokens")


def _units(inputs, o):
    budget = o["token_budget"]
    units = []
    for i, (content, questions) in enumerate(inputs):
        content = tuple(content)
        sizes = [question_size(q[0], q[1]) for q in questions]
        total = len(content) + sum(sizes)
        if total <= budget:
            units.append(Unit(i, list(range(len(questions))), content, [_norm(q) for q in questions], size=total))
            continue
        # long input: chunks of the full content plus a greedy run of questions
        j = 0
        if len(questions) == 0:
            raise PlanError("LIMIT", f"input {i}: content does not fit the token budget")
        while j < len(questions):
            size = len(content)
            held = []
            while j < len(questions) and size + sizes[j] <= budget:
                size += sizes[j]
                held.append(j)
                j += 1
            if not held:
                raise PlanError("LIMIT", f"input {i}: content plus question {j} do not fit the token budget")
            units.append(Unit(i, held, content, [_norm(questions[q]) for q in held], size=size))
    if o["floors"]:
        prefix = tuple(o["floor_prefix"])
        seen = {}
        for content, questions in inputs:
            for question in questions:
                if is_searched(question):
                    continue
                template, options = question
                k = _key(template, options)
                if k in seen:
                    continue
                seen[k] = True
                size = len(prefix) + question_size(template, options)
                if size > budget:
                    raise PlanError("LIMIT", "a floor input does not fit the token budget")
                units.append(Unit(-1, [0], prefix, [(tuple(template), [tuple(x) for x in options])],
                                  floor_key=k, size=size))
    return units


def _norm(question):
    """A question as tuples: ``(template, [options])`` or ``(template, None, token_set)``."""
    if is_searched(question):
        return (tuple(question[0]), None, int(question[2]))
    return (tuple(question[0]), [tuple(x) for x in question[1]])


def _pack(units, budget):
    """Next-fit: keep filling the current pass while the running total fits."""
    passes, cur, total = [], [], 0
    for u in units:
        if cur and total + u.size > budget:
            passes.append(cur)
            cur, total = [], 0
        cur.append(u)
        total += u.size
    if cur:
        passes.append(cur)
    return passes


def _layout_pass(units):
    tok, parent, content_lo, content_hi, chain, anchor = [], [], [], [], [], []
    records = []
    gather_rows, gather_tok = [], []
    x_rows, x_set = [], []
    for u in units:
        s = len(tok)
        u.start = s
        L = len(u.content)
        for i, t in enumerate(u.content):
            tok.append(t)
            parent.append(s + i - 1 if i > 0 else -1)
            content_lo.append(s)
            content_hi.append(s + i + 1)
            chain.append([])
            anchor.append(s)
        last_content = s + L - 1 if L > 0 else -1
        for qn, question in enumerate(u.questions):
            template, options = question[0], question[1]
            prev = last_content
            for t in template:
                r = len(tok)
                tok.append(t)
                parent.append(prev)
                content_lo.append(s)
                content_hi.append(s + L)
                chain.append((chain[prev] if prev >= s + L else []) + [r])
                anchor.append(s)
                prev = r
            slot = prev
            if options is None:   # searched slot: the template's last row is scored, nothing else is laid out
                records.append(QuestionRecord(u.source, u.qidx[qn], None, [], extract=len(x_rows)))
                x_rows.append(slot)
                x_set.append(question[2])
                continue
            node_row = {(): slot}
            for prefix in trie_nodes(options):
                r = len(tok)
                p = node_row[prefix[:-1]]
                tok.append(prefix[-1])
                parent.append(p)
                content_lo.append(s)
                content_hi.append(s + L)
                chain.append(chain[p] + [r])
                anchor.append(s)
                node_row[prefix] = r
            per_opt = []
            for opt in options:
                gs = []
                for i, t in enumerate(opt):
                    gs.append(len(gather_rows))
                    gather_rows.append(node_row[tuple(opt[:i])])
                    gather_tok.append(t)
                per_opt.append(gs)
            records.append(QuestionRecord(u.source, u.qidx[qn], _key(template, options), per_opt))
        u_end = len(tok)
        assert u_end - s == u.size
    T = len(tok)
    T_pad = -(-T // TILE) * TILE
    # pos = |visible set| - 1
    pos = [content_hi[q] - content_lo[q] + len(chain[q]) - 1 for q in range(T)]
    # end[k] = 1 + the largest row that sees k
    end = [k + 1 for k in range(T)]
    for q in range(T):
        for k in chain[q]:
            end[k] = max(end[k], q + 1)
    # content part: content rows below content_hi[q] are seen by q; suffix max
    # over content_hi gives, per content row, the largest row that sees it.
    for u in units:
        s, L = u.start, len(u.content)
        if L == 0:
            continue
        u_end = s + u.size
        best = [-1] * (L + 1)          # best[c]: largest q with content_hi - s == c
        for q in range(s, u_end):
            c = content_hi[q] - s
            best[c] = max(best[c], q)
        run = -1
        for c in range(L, 0, -1):      # content row s + c - 1 is seen by rows with hi >= c
            run = max(run, best[c])
            end[s + c - 1] = max(end[s + c - 1], run + 1)
    # pad rows
    for r in range(T, T_pad):
        tok.append(0)
        parent.append(-1)
        pos.append(0)
        end.append(r + 1)
        anchor.append(r)
    # schedule: per 128-row Q tile, per intersecting unit in layout order, the
    # unit-anchored KV tiles holding at least one key visible to a row of the tile;
    # a tile holds only the keys of its own unit (a key past the unit's end belongs
    # to the next unit and is read through that unit's own tiles)
    n_qt = T_pad // TILE
    tile_ptr = [0]
    tile_kv, tile_len = [], []
    for qt in range(n_qt):
        r0, r1 = qt * TILE, (qt + 1) * TILE
        for u in units:
            s, e = u.start, u.start + u.size
            lo, hi = max(r0, s), min(r1, e)
            if lo >= hi:
                continue
            hit = set()
            for q in range(lo, hi):
                if content_hi[q] > content_lo[q]:
                    hit.update(range(0, (content_hi[q] - 1 - s) // TILE + 1))
                for k in chain[q]:
                    hit.add((k - s) // TILE)
            for j in sorted(hit):
                tile_kv.append(s + TILE * j)
                tile_len.append(min(TILE, e - (s + TILE * j)))   # keys of the tile inside this input
        tile_ptr.append(len(tile_kv))
    rows = sorted(set(gather_rows) | set(x_rows))
    m_of = {r: m for m, r in enumerate(rows)}
    i32 = lambda a: np.asarray(a, dtype=np.int32)  # noqa: E731
    return PassLayout(
        T=T, T_pad=T_pad, tok=i32(tok), parent=i32(parent), pos=i32(pos), end=i32(end), anchor=i32(anchor),
        tile_ptr=i32(tile_ptr), tile_kv=i32(tile_kv), tile_len=i32(tile_len), slot_row=i32(rows),
        gather_m=i32([m_of[r] for r in gather_rows]), gather_tok=i32(gather_tok),
        x_m=i32([m_of[r] for r in x_rows]), x_set=i32(x_set),
        units=units, questions=records,
        content_lo=i32(content_lo), content_hi=i32(content_hi), chain=chain,
    )


def plan(inputs, **opts) -> Plan:
    """Lay ``inputs`` out in packed passes.

    ``inputs`` is a list of ``(content_ids, [question, ...])`` or
    ``(content_ids, [question, ...], [grid, ...])``, a question being
    ``(template_ids, [option_ids, ...])`` or, for a searched slot,
    ``(template_ids, None, token_set)``, and a grid
    ``(segments, values, options)`` or ``(segments, values, None, token_set)``.
    Options are keyword arguments named as in :data:`DEFAULTS`.
    """
    o = dict(DEFAULTS)
    unknown = set(opts) - set(o)
    if unknown:
        raise TypeError(f"unknown options {sorted(unknown)}")
    o.update(opts)
    inputs = _expand_inputs(inputs, o)
    _validate(inputs, o)
    units = _units(inputs, o)
    passes = [_layout_pass(us) for us in _pack(units, o["token_budget"])]
    question_home, floor_home = {}, {}
    for p, lay in enumerate(passes):
        for idx, rec in enumerate(lay.questions):
            if rec.source >= 0:
                question_home[(rec.source, rec.qidx)] = (p, idx)
            else:
                floor_home[rec.key] = (p, idx)
    return Plan(
        passes=passes,
        n_inputs=len(inputs),
        n_questions=[len(q) for _, q in inputs],
        n_options=[[0 if is_searched(x) else len(x[1]) for x in q] for _, q in inputs],
        searched=[[is_searched(x) for x in q] for _, q in inputs],
        extract_k=o["extract_k"],
        question_home=question_home,
        floor_home=floor_home,
    )
