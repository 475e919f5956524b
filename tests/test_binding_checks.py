"""The Python binding's argument checks, which run before the library is
called: wrong dtypes, host tensors and mismatched shapes raise at once, so a
caller never reaches the C ABI with a tensor it cannot take (no GPU needed)."""

import pytest
import torch

from tiled_attention_attn_gb300 import attn


def t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def test_forward_rejects_float32_and_mixed_dtypes():
    with pytest.raises(TypeError):
        attn.attn_fwd(t(1, 8, 2, 64, dtype=torch.float32), t(1, 8, 2, 64), t(1, 8, 2, 64))
    with pytest.raises(TypeError):
        attn.attn_fwd(t(1, 8, 2, 64), t(1, 8, 2, 64, dtype=torch.float16), t(1, 8, 2, 64))


def test_forward_rejects_host_tensors():
    with pytest.raises(ValueError):
        attn.attn_fwd(t(1, 8, 2, 64), t(1, 8, 2, 64), t(1, 8, 2, 64))


def test_backward_rejects_mixed_dtypes_and_host_tensors():
    q = t(1, 8, 2, 64)
    with pytest.raises(TypeError):
        attn.attn_bwd(q, q, q, q, torch.zeros(1, 2, 8), t(1, 8, 2, 64, dtype=torch.float16))
    with pytest.raises(ValueError):
        attn.attn_bwd(q, q, q, q, torch.zeros(1, 2, 8), q)


def test_decode_rejects_bad_dtypes_and_host_tensors():
    q, k = t(2, 4, 64), t(10, 2, 64)
    cu = torch.tensor([0, 5, 10], dtype=torch.int32)
    with pytest.raises(TypeError):
        attn.attn_decode(q.float(), k, k, cu)
    with pytest.raises(ValueError):
        attn.attn_decode(q, k, k, cu)                      # host tensors
