"""Float64 CPU oracle for exact tiled attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import anything from this package.  The CUDA
library and its Python binding never import it, and it imports nothing from
them: the two sides share no code.

Pages this package follows (cited by title and section throughout):

* "Flash attention and efficient attention -- Hinglish notes" (4.1.14,
  AI-ML > Transformer Architecture), called NOTES below: sections
  "The Standard Attention Problem", "Derivation: Incremental Softmax"
  (Steps 1-3), "Worked example Flash Attention Forward Pass (Simplified)",
  "Backward Pass: Recomputation", "Worked example Local Attention Window".
* "Compute attention one tile at a time" (TensorViz flash-attention teaching
  example), called TVIZ below: steps "dense", "coupled", "tiles",
  "equivalent", its numerical-check list and the tile replay experiment.

Every function is pinned by a ``-m "not gpu"`` test against something other
than itself (printed values from the pages, closed forms, invariants, library
routines, finite differences); see ``tests/test_oracle_*.py``.  No function
here is "parity unpinned".
"""

from .attention import (  # noqa: F401
    NEG_INF,
    window_radius,
    window_mask,
    dense_scores,
    dense_forward,
    dense_forward_rows,
    banded_forward_rows,
    block_statistics,
    merge_statistics,
    tiled_forward,
    dense_backward,
)
