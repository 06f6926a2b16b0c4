"""GB300-native (sm_103a) grouped-query attention.

Two hot paths behind a C ABI (include/attn.h, libattn_gb300.so):

* ``attn_prefill``      causal / full GQA prefill on tcgen05 tensor cores
* ``attn_decode_paged`` single-token decode over a paged KV cache
  (split-K main kernel + log-sum-exp combine kernel)

This package is the thin Python binding: PyTorch provides device memory and
streams, the library does all of the work.
"""
from ._binding import (  # noqa: F401
    ATTN_ERR_BAD_INPUT,
    ATTN_ERR_CUDA,
    ATTN_ERR_INVALID_ARG,
    ATTN_ERR_TIMEOUT,
    ATTN_ERR_UNSUPPORTED,
    ATTN_ERR_WORKSPACE,
    ATTN_OK,
    EXPORTED,
    NOALLOC_SCRATCH_BYTES,
    AttnError,
    attn_debug_prefill_stall,
    attn_decode_paged,
    attn_decode_paged_append,
    attn_decode_paged_noalloc,
    attn_kv_append,
    attn_decode_paged_workspace_bytes,
    attn_decode_paged_ws,
    attn_get_device_error,
    attn_lse_combine,
    attn_prefill,
    attn_prefill_paged,
    attn_release_workspace,
    attn_version,
    load,
    status_string,
)
