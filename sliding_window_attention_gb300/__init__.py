"""GB300 (sm_103a) causal / sliding-window grouped-query attention.

The compute lives in libswa_attn.so (C ABI, include/swa_attn.h); this
package is its thin Python binding plus the seeded input generators.
The library is loaded on first use and every call fails loudly if it is
missing: there is no CPU fallback.
"""
from ._native import (  # noqa: F401
    SwaError,
    backward,
    bwd_workspace_bytes,
    bwd_workspace_bytes_ex,
    bwd_workspace_bytes_prefix,
    forward,
    fwd_workspace_bytes,
    fwd_workspace_bytes_ex,
    fwd_workspace_bytes_prefix,
    load,
    profile_begin,
    profile_end,
    strerror,
    swa_attn_bwd,
    swa_attn_bwd_ex,
    swa_attn_bwd_prefix,
    swa_attn_bwd_sinks,
    swa_attn_fwd,
    swa_attn_fwd_ex,
    swa_attn_fwd_prefix,
    swa_attn_fwd_sinks,
    swa_attn_get_status,
    swa_attn_selftest_timeout,
)

__all__ = [
    "SwaError", "backward", "bwd_workspace_bytes", "bwd_workspace_bytes_ex", "forward", "fwd_workspace_bytes",
    "fwd_workspace_bytes_ex", "load", "profile_begin", "profile_end", "strerror", "swa_attn_bwd", "swa_attn_bwd_ex",
    "swa_attn_fwd", "swa_attn_fwd_ex", "swa_attn_get_status", "swa_attn_selftest_timeout",
    "fwd_workspace_bytes_prefix", "bwd_workspace_bytes_prefix", "swa_attn_fwd_prefix", "swa_attn_bwd_prefix",
    "swa_attn_fwd_sinks", "swa_attn_bwd_sinks",
]
