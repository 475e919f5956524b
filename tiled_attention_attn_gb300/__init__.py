"""GB300 (sm_103a) tiled attention forward: O = softmax(scale * Q K^T [+ causal]) V
with online-softmax running statistics, and its backward (dq, dk, dv from the
kept lse), behind the C ABI of include/attn.h.

The binding loads libattn.so on first use; build it with
``tiled_attention_attn_gb300.build.build()``.
"""

from .attn import (  # noqa: F401
    AttnError,
    attn_bwd,
    attn_decode,
    attn_func,
    attn_func_padded,
    attn_fwd,
    get_error,
    last_device_error,
    lib,
    plan,
    selftest_wait_timeout,
    set_wait_timeout_ns,
    strerror,
)
