"""GB300 paged attention and greedy speculative verification.

A thin Python binding over the C ABI in include/specattn.h (libspecattn.so):
it marshals torch tensors to pointers and returns the library's status codes
as exceptions. Every step of the computation runs in the library's CUDA
kernels; there is no Python or CPU fallback, and importing the package does
not build anything (``speculative_decode_gb300.build.build()`` does).
"""
from ._lib import (  # noqa: F401
    Dims,
    Plan,
    SpecAttnError,
    STATUS,
    defrag_apply,
    defrag_apply_bytes,
    defrag_moves,
    dims_for,
    kv_append,
    kv_append_q4,
    kv_append_q8,
    library_path,
    load_library,
    paged_attn,
    paged_attn_q4,
    paged_attn_q8,
    paged_attn_kernel_count,
    paged_attn_noalloc,
    paged_attn_workspace_size,
    plan_analyze,
    selftest_bounded_wait,
    sm_count,
    spec_verify_greedy,
    spec_verify_greedy_advance,
    spec_verify_workspace_size,
    status_string,
)
