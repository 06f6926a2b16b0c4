"""GB300-native (sm_103a) grouped-query attention.

Two hot paths behind a C ABI (include/attn.h, libattn_gb300.so):

* ``attn_prefill``      causal / full GQA prefill on tcgen05 tensor cores
* ``attn_decode_paged`` single-token decode over a paged KV cache
  (split-K main kernel + log-sum-exp combine kernel)
* ``attn_prefill_paged`` chunked prefill of new query chunks over the paged
  cache (cached prefixes, ragged lengths)
* ``attn_kv_append`` / ``attn_qk_norm_rope(_append)`` the attention-input
  prologue: KV append, per-head QK-norm and NeoX RoPE

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
    attn_prefill_paged_qk_norm_rope,
    attn_qk_norm_rope,
    attn_qk_norm_rope_append,
    attn_rope_cos_sin_table,
    attn_release_workspace,
    attn_version,
    load,
    status_string,
)
