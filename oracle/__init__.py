"""Plain CPU oracle for the vocabulary-wide hot path of block speculative decoding.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline and
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code, constant
table or helper with the CUDA library in ``verify_spec_draft_gb300/csrc``; the two
meet only in the seeded input generators (``verify_spec_draft_gb300.synth``), which
hold none of the method's arithmetic.

Every value is computed in float64 (bf16 inputs widen exactly).  The functions follow
the pages step by step, in their order and notation:

* ``philox``  - Philox4x64-10 counter RNG (Salmon et al., SC'11) and the 24-bit uniform
  that both sides draw.
* ``draft``   - the DSpark block draft: low-rank Markov bias W_1[x_{j-1}] W_2 added to
  each position's logits, softmax, argmax or inverse-CDF sample, confidence.
* ``verify``  - target verification of a draft block: longest argmax-matching prefix
  (T=0) or rejection sampling with a residual/bonus draw (T=1).
* ``e2etv``   - the SpecOPD E2E-TV surrogate: overlap 1-TV, prefix survival products,
  their mean, and the gradient with respect to the draft logits.
* ``anchors`` - the SpecOPD anchor-branch plan: distinct random anchors on each
  reference response, the anchor tokens, and the parent map and semantic positions
  that pack the drafted branches into one proposal tree.
* ``topk``    - top-k / top-p filtered sampling at T=1 (the DSpine card's setting) for
  the draft's draws and the target's verification.
* ``tree``    - EAGLE-2 draft trees: path-product scores, the prefix-closed top-m
  selection, and T=0 verification along the tree's paths.
* ``schedule`` - the DSpark verify budget: per-request pass products of the confidences,
  the budget given to the most likely positions across the batch, the throughput
  against a cost curve.

Pins (tests that tie each function to the pages or to mathematics rather than to
itself) live in ``tests/test_oracle_*.py``; each function's docstring names them.
"""

from . import philox, draft, verify, e2etv, schedule, anchors, topk, tree  # noqa: F401
