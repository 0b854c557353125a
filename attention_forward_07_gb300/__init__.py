"""GB300-native (sm_103a) fused attention forward.

``O = softmax(scale * Q K^T + mask) V`` and the row log-sum-exp, computed tile by
tile with an online softmax by hand-written CUDA kernels (TMA, mbarrier,
tcgen05.mma with TMEM accumulators) behind the C-ABI declared in
``include/attn.h``.  This package is the thin Python binding over that library
(argument marshalling only); importing it does not load the library, calling
into it does, and a missing or unloadable library raises -- there is no CPU
fallback.
"""
from ._binding import (  # noqa: F401
    ATTN_BF16,
    ATTN_F16,
    AttnError,
    attn_check,
    attn_fwd,
    attn_fwd_ex,
    attn_fwd_noalloc,
    attn_fwd_packed,
    attn_fwd_visited,
    attn_release_workspace,
    attn_strerror,
    attn_tile_shape,
    debug_counters,
    library,
    library_path,
)
