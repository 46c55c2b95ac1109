"""Float64 CPU oracle for the EntmaxKV decode step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package. The product path (the CUDA library and its Python
binding) never calls into it, and this package never imports the product.

What it computes follows "EntmaxKV: Support-Aware Decoding for Entmax
Attention" (gist.science technical summary, §2 A-C and §3; arXiv abstract on
the mlsanity.com index page). Every function says which passage it follows.
Where the pages leave a step open, the reading taken is stated in the
function's docstring.

Modules:
  entmax  -- α-entmax threshold and probabilities (exact), softmax.
  pages   -- per-page metadata, bounding-box bound, Gaussian page model,
             the normalisation solve for τ̂, top-k and Gaussian selection.
  decode  -- one decode step per (sequence, KV head): selection, sparse
             entmax attention, τ, dropped mass δ, support recall.

Pins: the pages print no worked example and no numeric value for τ, τ̂, δ,
recall or outputs on any input, so no function here is checked against a
printed number. Every function is pinned instead by closed forms, textbook
special cases, brute force on small inputs and the invariants the pages
state; ``tests/test_oracle_*.py`` hold those pins.
"""

from . import entmax, pages, decode  # noqa: F401
