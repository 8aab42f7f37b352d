"""GB300-native fused attention forward and backward (sm_103a).

The compute path is the C-ABI library ``libattn_fwd.so`` built from ``csrc/``;
``attn_fwd`` and friends (in ``binding``) only marshal arguments to it.  The
library is loaded on first use, and any failure to load it is an error: there
is no fallback path.
"""
from .binding import (  # noqa: F401
    AttnError,
    attn_bwd,
    attn_bwd_varlen,
    attn_fwd,
    attn_fwd_fp8,
    attn_fwd_host,
    attn_fwd_kvcache,
    attn_fwd_kvcache_paged,
    attn_fwd_splitkv,
    attn_fwd_varlen,
    bwd_workspace_bytes,
    lib_path,
    load,
    status,
)
