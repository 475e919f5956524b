"""Parity of attn_fwd_rope (the forward of rotary-embedded queries and keys,
the rotation of Q fused into the forward kernel) with the fp64 oracle, through
the C ABI.

Reference: the oracle's rotary (training page §4: pair p of the first rot_dim
features rotated by position * base^(-2p/rot_dim), GPT-NeoX or GPT-J pairing)
applied to q at positions q_offset + i and to k at positions j, each rotated
tensor rounded to the inputs' 16-bit type (as the library stores the rotated
values), then the oracle's attention.  Bars as in test_parity_gpu: max
|O - O_ref| <= 1e-2, max |lse - lse_ref| <= 1e-3.  Also compared with the
unfused route (attn_rotary on q and k, then attn_fwd) on the same inputs.
"""

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    return attn_lib


def rotated(x, positions, rot, base, interleaved):
    """oracle rotary of x (B, L, H, d) with one position per token, rounded to x's dtype"""
    B, L, H, d = x.shape
    flat = x.reshape(B * L, H, d)
    pos = np.tile(np.asarray(positions), B)
    r = oracle.rotary(flat, pos, rot, base, interleaved)
    return torch.from_numpy(r).to(x.dtype).reshape(B, L, H, d)


CASES = [
    # B, Hq, Hkv, Lq, Lk, d, dtype, causal, rot, interleaved, q_offset
    (1, 2, 2, 300, 300, 128, torch.bfloat16, True, 128, False, 0),
    (2, 4, 2, 257, 257, 128, torch.bfloat16, False, 64, True, 0),
    (1, 4, 1, 100, 700, 64, torch.float16, True, 32, False, 600),    # queries after a cache
    (1, 8, 8, 129, 129, 64, torch.bfloat16, True, 64, True, 0),
    (1, 1, 1, 4096, 4096, 128, torch.bfloat16, True, 128, False, 0),  # split pieces merged
    (2, 2, 2, 1, 1, 128, torch.float16, False, 16, False, 5),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_rope_fused_matches_oracle(case):
    B, Hq, Hkv, Lq, Lk, d, dtype, causal, rot, inter, qoff = case
    g = torch.Generator().manual_seed(B * 1000 + Lq + rot)
    q = torch.randn(B, Lq, Hq, d, generator=g).to(dtype)
    k = torch.randn(B, Lk, Hkv, d, generator=g).to(dtype)
    v = torch.randn(B, Lk, Hkv, d, generator=g).to(dtype)
    dev = torch.device("cuda", 0)
    scale = d ** -0.5
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = attn.attn_fwd_rope(qd, kd, vd, causal=causal, scale=scale, rot_dim=rot, base=10000.0,
                                interleaved=inter, q_offset=qoff)
    assert attn.get_error() == attn.ATTN_OK
    # q and k are left as they were
    assert torch.equal(qd.cpu(), q) and torch.equal(kd.cpu(), k)
    qr = rotated(q, np.arange(Lq) + qoff, rot, 10000.0, inter)
    kr = rotated(k, np.arange(Lk), rot, 10000.0, inter)
    if Lq * Lk <= 300 * 700 * 4:
        o_ref, lse_ref = oracle.attention(qr, kr, v, causal=causal, scale=scale)
        on = o.float().cpu().double().numpy()
        ln = lse.cpu().double().numpy()
    else:
        rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in np.linspace(0, Lq - 1, 96).astype(int)]
        o_ref, lse_ref = oracle.attention_rows(qr, kr, v, rows, causal=causal, scale=scale)
        idx = np.array(rows)
        on = o.float().cpu().double().numpy()[idx[:, 0], idx[:, 2], idx[:, 1]]
        ln = lse.cpu().double().numpy()[idx[:, 0], idx[:, 1], idx[:, 2]]
    assert float(np.abs(on - o_ref).max()) <= O_TOL
    assert float(np.abs(ln - lse_ref).max()) <= LSE_TOL


@pytest.mark.parametrize("interleaved", [False, True])
def test_rope_fused_agrees_with_the_unfused_route(interleaved):
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(9)
    q = torch.randn(2, 1000, 8, 128, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(2, 1000, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(2, 1000, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    o1, l1 = attn.attn_fwd_rope(q, k, v, causal=True, rot_dim=128, interleaved=interleaved)
    qr = attn.rotary(q, rot_dim=128, interleaved=interleaved)
    kr = attn.rotary(k, rot_dim=128, interleaved=interleaved)
    o2, l2 = attn.attn_fwd(qr, kr, v, causal=True)
    assert attn.get_error() == attn.ATTN_OK
    assert float((o1.float() - o2.float()).abs().max()) <= O_TOL
    assert float((l1 - l2).abs().max()) <= LSE_TOL


def test_rope_fused_rejects_bad_rotary_arguments():
    dev = torch.device("cuda", 0)
    q = torch.randn(1, 16, 2, 64, device=dev, dtype=torch.bfloat16)
    for kw in (dict(rot_dim=24), dict(rot_dim=80), dict(base=1.0), dict(q_offset=-1)):
        with pytest.raises(attn.AttnError):
            attn.attn_fwd_rope(q, q, q, **kw)
