"""Float64 CPU oracle (test infrastructure only; see sink_attention.py).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  The CUDA library never does, and this package never imports
the CUDA library.
"""
from .sink_attention import (  # noqa: F401
    attend_rows,
    decode,
    decode_multi,
    gather_paged_kv,
    online_split_merge,
    paged_attention,
    prefill,
    prefill_rows,
    sink_softmax_rows,
)
from .rope import qkv_bias_rope, rope, yarn_inv_freq  # noqa: F401
