"""GB300-native grouped-query attention with a per-head attention sink.

Python face of the C-ABI library libsink_attn.so (see include/sink_attn.h):
causal variable-length prefill, split-KV paged decode, multi-token decode,
chunked prefill (new tokens per sequence against the paged cache), and the
QKV bias + YaRN rotary pass that prepares q, k and v (and appends k and v to
the cache).  The functions only
marshal torch tensors into the C calls; all the arithmetic runs in the CUDA
kernels, and a missing library is an error, never a fallback.
"""
from .binding import (  # noqa: F401
    OUT_BF16,
    OUT_F32,
    SinkAttnError,
    load,
    sink_attn_decode,
    sink_attn_decode_max_splits,
    sink_attn_decode_multi,
    sink_attn_decode_multi_workspace_bytes,
    sink_attn_decode_noalloc,
    sink_attn_decode_rope,
    sink_attn_decode_workspace_bytes,
    sink_attn_get_device_error,
    sink_attn_prefill,
    sink_attn_prefill_paged,
    sink_attn_prefill_paged_workspace_bytes,
    sink_attn_prefill_rope,
    sink_attn_qkv_rope,
    sink_attn_status_string,
    sink_attn_version,
    sink_attn_yarn_inv_freq,
)
