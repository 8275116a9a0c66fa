"""GB300-native streaming attention forward.

The compute path is the C-ABI shared library built from ``csrc/``; the
Python functions in ``binding`` only marshal arguments to it. Importing this
package does not load the library: the first call does, and it raises if the
library has not been built.
"""
from .binding import (  # noqa: F401
    ATTN_BF16,
    ATTN_FP16,
    ATTN_FP32,
    PATH_AUTO,
    PATH_DECODE,
    PATH_PREFILL,
    PATH_PREFILL_PAIR,
    PATH_SIMT,
    AttnError,
    attention,
    attention_fp8,
    attention_lse,
    attn_bwd,
    attn_bwd_workspace_bytes,
    attn_decode_paged,
    attn_decode_paged_fp8,
    attn_decode_paged_fp8_workspace_bytes,
    attn_decode_paged_workspace_bytes,
    attn_fwd,
    attn_fwd_decode_noalloc,
    attn_fwd_ex,
    attn_fwd_ws,
    attn_fwd_fp8,
    attn_fwd_fp8_workspace_bytes,
    attn_fwd_host,
    attn_fwd_lse,
    attn_merge,
    attn_split_softmax_workspace_bytes,
    attn_workspace_bytes,
    attn_workspace_bytes_ex,
    last_device_status,
    lib,
    selftest_bounded_wait,
    selftest_prefill_abort,
    split_softmax,
    library_path,
    strerror,
)
