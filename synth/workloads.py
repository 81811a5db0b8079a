"""Request structures shaped like the pages' workloads (inputs only).

An input is ``(content_ids, [(template_ids, [option_ids, ...]), ...])``.  Token
ids are uniform in ``[0, vocab)``; the options of one question are distinct.

The pages' own workloads (a public 24-article news fixture with 56 two-option
questions each, a 106-question moderation pack, extraction-heavy jobs) are not
available; these seeded structures stand in for them with the sizes the pages
state ("spinf-serve 0.1.1" PyPI page, "Speed and scale"; "spinf-serve" man page,
PARAMETERS).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Shape:
    """Attention and lm-head shape of one workload."""

    n_q_heads: int
    n_kv_heads: int
    d_head: int
    d_model: int
    vocab: int
    window: int = 0          # sliding window of the windowed layer variant (0: none)


TINY = Shape(4, 2, 64, 256, 1024)
GEMMA = Shape(16, 8, 256, 3840, 262144)
GEMMA_WINDOWED = Shape(16, 8, 256, 3840, 262144, window=1024)
QWEN = Shape(40, 8, 128, 5120, 151936, window=1024)


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _ids(g, n, vocab):
    return [int(x) for x in g.integers(0, vocab, size=n)]


def _distinct(g, n, vocab):
    return [int(x) for x in g.choice(vocab, size=n, replace=False)]


def _two_option_questions(g, n, lo, hi, vocab, n_opts=(2, 2)):
    qs = []
    for _ in range(n):
        k = int(g.integers(n_opts[0], n_opts[1] + 1))
        qs.append((_ids(g, int(g.integers(lo, hi + 1)), vocab), [[t] for t in _distinct(g, k, vocab)]))
    return qs


def tiny(seed=0, vocab=1024):
    """2 contents of 64 tokens, 4 questions of 8 tokens each, 2 single-token options."""
    g = _rng(seed)
    return [(_ids(g, 64, vocab), _two_option_questions(g, 4, 8, 8, vocab)) for _ in range(2)]


def wikinews(seed=0, vocab=262144, n_contents=24, n_questions=56):
    """24 contents of U[400, 540] tokens sharing one set of 56 two-option questions of U[8, 16] tokens."""
    g = _rng(seed)
    questions = _two_option_questions(g, n_questions, 8, 16, vocab)
    return [(_ids(g, int(g.integers(400, 541)), vocab), questions) for _ in range(n_contents)]


#: messages that fill exactly three 16384-token passes, floors included (seed 0)
MODERATION_MESSAGES = 23


def moderation(seed=0, vocab=262144, n_messages=MODERATION_MESSAGES):
    """Messages of U[30, 200] tokens sharing one set of 106 questions of U[10, 24] tokens, 2-3 options."""
    g = _rng(seed)
    questions = _two_option_questions(g, 106, 10, 24, vocab, n_opts=(2, 3))
    return [(_ids(g, int(g.integers(30, 201)), vocab), questions) for _ in range(n_messages)]


def _prefix_free_options(g, vocab):
    """2-5 options of 1-3 tokens, no option a prefix of another; some share first tokens."""
    while True:
        n = int(g.integers(2, 6))
        opts = []
        for _ in range(n):
            L = int(g.integers(1, 4))
            if opts and L > 1 and g.random() < 0.5:
                base = opts[int(g.integers(0, len(opts)))]
                opt = [base[0]] + _ids(g, L - 1, vocab)
            else:
                opt = _ids(g, L, vocab)
            opts.append(opt)
        tup = [tuple(o) for o in opts]
        ok = len(set(tup)) == len(tup) and not any(
            a != b and b[:len(a)] == a for a in tup for b in tup)
        if ok:
            return opts


def stress(seed=0, vocab=151936, n_questions=1000, content_tokens=4000):
    """1 content of 4000 tokens, 1000 questions of U[10, 20] tokens with 2-5 options of 1-3 tokens."""
    g = _rng(seed)
    content = _ids(g, content_tokens, vocab)
    qs = [(_ids(g, int(g.integers(10, 21)), vocab), _prefix_free_options(g, vocab)) for _ in range(n_questions)]
    return [(content, qs)]


def invariance_target(seed=0, vocab=262144):
    """A 470-token content with 56 two-option questions of U[8, 16] tokens."""
    g = _rng(seed + 1000)
    return (_ids(g, 470, vocab), _two_option_questions(g, 56, 8, 16, vocab))


def short_inputs(seed=0, vocab=262144, n=2000):
    """Short inputs: content U[8, 40], 1-4 two-option questions of U[8, 16] tokens."""
    g = _rng(seed + 2000)
    return [(_ids(g, int(g.integers(8, 41)), vocab),
             _two_option_questions(g, int(g.integers(1, 5)), 8, 16, vocab)) for _ in range(n)]


def invariance_packing(packing_seed, seed=0, vocab=262144, n_short=2000):
    """The target inserted at a uniformly random index among the short inputs.

    Returns ``(inputs, target_index)``.
    """
    target = invariance_target(seed, vocab)
    shorts = short_inputs(seed, vocab, n_short)
    idx = int(_rng(packing_seed).integers(0, len(shorts) + 1))
    return shorts[:idx] + [target] + shorts[idx:], idx


def with_searched_slots(inputs, n, seed=0, vocab=262144, n_sets=2):
    """Every input gets the same ``n`` searched slots appended to its questions:
    templates of U[8, 16] tokens, token sets cycling -1 (any token), 0, 1, ...,
    ``n_sets - 1`` (a question is then ``(template, None, token_set)``)."""
    g = _rng(seed + 3000)
    slots = [(_ids(g, int(g.integers(8, 17)), vocab), None, (i % (n_sets + 1)) - 1) for i in range(n)]
    return [(content, list(questions) + slots) for content, questions in inputs]


def token_sets(vocab, n_sets=2, density=0.01, seed=0):
    """Allowed-token sets of searched slots (stand-ins for a tokenizer's digit and
    amount tokens): ``[n_sets, vocab]`` booleans, each a seeded random ``density``
    fraction of the vocabulary, plus the last token (the ragged end of the vocabulary)."""
    g = _rng(seed + 4000)
    out = g.random((n_sets, vocab)) < density
    out[:, vocab - 1] = True
    return out


def invariance(seed=0, vocab=262144, packing_seed=1):
    """One packing of the batch-invariance pass as a request: 2000 short inputs with the
    470-token target inserted at a random index (its lm head is e4m3 in the benchmarks)."""
    return invariance_packing(packing_seed, seed, vocab)[0]


def wikinews_grid(seed=0, vocab=262144, n_contents=24):
    """The Wikinews-shaped job with its questions as one placeholder grid per content: literal
    pieces of 4, 3 and 2 tokens around two placeholders of 7 and 8 values (1-2 tokens each),
    two single-token options: 56 cells of 11-13 tokens per content.  A grid is
    ``(pieces, values per placeholder, options)``; the input is ``(content, [], [grid])``."""
    g = _rng(seed + 5000)
    pieces = [_ids(g, 4, vocab), _ids(g, 3, vocab), _ids(g, 2, vocab)]
    values = [[_ids(g, int(g.integers(1, 3)), vocab) for _ in range(7)],
              [_ids(g, int(g.integers(1, 3)), vocab) for _ in range(8)]]
    grid = (pieces, values, [[t] for t in _distinct(g, 2, vocab)])
    return [(_ids(g, int(g.integers(400, 541)), vocab), [], [grid]) for _ in range(n_contents)]


def written_out(inputs):
    """The same inputs with every grid cell written out as a question, first placeholder
    slowest (the order a grid's cells take in the plan)."""
    out = []
    for content, questions, *rest in inputs:
        qs = list(questions)
        for grid in (rest[0] if rest else []):
            pieces, values, options, tail = grid[0], grid[1], grid[2], tuple(grid[3:])   # tail: a searched token set

            def cells(i, acc):
                if i == len(values):
                    yield acc + pieces[-1]
                    return
                for val in values[i]:
                    yield from cells(i + 1, acc + pieces[i] + val)
            qs.extend((tmpl, options, *tail) for tmpl in cells(0, []))
        out.append((content, qs))
    return out


WORKLOADS = {
    "tiny": (tiny, TINY),
    "wikinews": (wikinews, GEMMA),
    "moderation": (moderation, GEMMA_WINDOWED),
    "stress": (stress, QWEN),
    "invariance": (invariance, GEMMA),
}
