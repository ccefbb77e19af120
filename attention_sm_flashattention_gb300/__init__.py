"""GB300 FlashAttention: exact tiled attention forward and backward for sm_103a.

``fwd``/``bwd`` call the C ABI of ``libfa.so`` (built in-tree by
``attention_sm_flashattention_gb300.build``).  The library is loaded on the
first call; if it is missing the call raises -- there is no other path.
"""

from .api import bwd, bwd_flops, bwd_workspace_size, device_status, fwd, fwd_flops, fwd_paged, fwd_sparse, paged_split_count, reshape_and_cache  # noqa: F401
