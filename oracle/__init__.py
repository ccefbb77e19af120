"""fp64 CPU oracle for exact softmax attention (test infrastructure only).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does.
"""

from .attention import (  # noqa: F401
    attn_bwd_head,
    attn_bwd_ref,
    attn_fwd_head,
    attn_fwd_ref,
    causal_tile_count,
    scores,
    softmax_probs,
)
