"""Oracle: a plain, slow, fp64 CPU restatement of the branch-packed scoring hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
anything under this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It shares
no code, table or constant generator with ``branch_packed_scoring_gb300``: it is an
independent reading of the pages, written so that a reader can check it against
them by eye.

Sources (web pages, cited by title and section):

* "spinf-serve 0.1.1" (PyPI project page), sections "What it does",
  "Speed and scale", "Install and run" -- the method: a content is read once,
  every question is a branch of the same pass that sees its own content and
  itself, never a sibling or another packed input; scores are per-option
  log-probabilities, ``p`` renormalised over the options, the floor (same
  question on empty content) and the residual mass.
* "spinf-serve" man page (linuxcommandlibrary), PARAMETERS and CAVEATS -- the
  16384-token pass budget and the per-input limits; long inputs run alone.
* "spinf-serve" news repost (aitujian.cn), English part -- the worked
  example of one two-option question (logprob, p, floor_p, residual).

Modules:

* :mod:`oracle.plan`      -- layout of inputs into packed passes (integer work).
* :mod:`oracle.attention` -- tree-masked softmax attention in fp64.
* :mod:`oracle.score`     -- vocabulary log-softmax at slot rows in fp64.
* :mod:`oracle.collect`   -- per-option log-prob, p, residual and floor.
* :mod:`oracle.fp8`       -- the e4m3 number format, from its definition.

Every function is pinned by ``tests/test_oracle_*.py`` to something other than
itself (brute force on unpacked sequences, closed forms, library routines,
the worked example).  The only function without such a pin is noted in its
docstring ("parity unpinned").
"""
