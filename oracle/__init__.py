"""fp64 CPU oracle for the attention forward pass (test infrastructure only)."""

from .oracle import attn_bwd, attn_fwd, attn_rows, build, default_threads, merge_proj, proj_heads  # noqa: F401
