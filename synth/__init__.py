"""Seeded synthetic inputs for the branch-packed scoring path.

This package holds no arithmetic of the method.  It only makes inputs:

* :mod:`synth.workloads` -- request structures (contents, question templates,
  option lists as token ids) shaped like the pages' workloads;
* :mod:`synth.values` -- activations and lm-head weights drawn from a
  counter-based generator keyed by each token's root path, so a token's values
  depend on its logical prefix and never on where it was packed.

Both the oracle tests and the CUDA path take their inputs from here.
"""
