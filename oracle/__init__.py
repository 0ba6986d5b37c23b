"""CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE, not product code.

This package is a plain, slow, float64 restatement of what the attention hot path
computes.  It exists only so that tests can check the CUDA kernels against an
independent implementation.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / ``--impl reference`` leg may import it.  The product
path (``online_softmax_14_b300``) never imports, links or calls anything here, and
nothing here imports the product path: the two share no code.

Modules
-------
attention
    The definition: materialise the N x N score matrix, mask it, two-pass safe
    softmax, weight the values (forward), and the textbook softmax-attention
    gradient (backward).
online
    A model of the tiled one-pass algorithm -- the running max / normaliser /
    accumulator recurrence and the block-state merge rule -- used to pin the
    definition against the pages' worked merges and to demonstrate that the
    rescale factor is required; and the same merge rule for normalised partial
    results (O_p, lse_p), the definition the split-key merge kernel is checked
    against.

Every function states the passage of the source pages it follows.  Parity of every
function here is pinned by ``tests/test_oracle_*.py`` against values the pages
print, closed forms, invariants and high-precision brute force.
"""

from .attention import (  # noqa: F401
    NEG_INF,
    STRICT,
    attention_bwd,
    attention_fwd,
    attention_fwd_rows,
    score_matrix,
)
from .online import merge_outputs, merge_states, online_attention, online_row  # noqa: F401
