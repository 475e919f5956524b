"""Parity of attn_rotary with the oracle's float64 rotary embedding, and of
rotary + the cache forward with the oracle's composition (training page §4,
new tokens starting at the cache length).  The kernel works in fp32 and rounds
to the tensor's 16-bit type.  Bar per feature, from that arithmetic: 1.5 units
in the last place of the reference, plus the fp32 rounding of the angle
(|a| 2^-21, a = position * frequency, covering the product and the frequency)
times the norm of the feature's pair; the attention bar is as elsewhere."""

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    return attn_lib


def ulp(ref, dtype):
    mant = 7 if dtype == torch.bfloat16 else 10
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
    return np.exp2(e - mant)


def angle_term(x, pos, rot, interleaved):
    """|a| 2^-21 times the pair norm, per feature (0 for unrotated features)."""
    x = oracle.f64(x)
    t = np.zeros_like(x)
    half = rot // 2
    for p in range(half):
        i1, i2 = (2 * p, 2 * p + 1) if interleaved else (p, p + half)
        a = np.abs(np.asarray(pos, np.float64) * 10000.0 ** (-2.0 * p / rot))[:, None]
        nrm = np.hypot(x[:, :, i1], x[:, :, i2])
        t[:, :, i1] = t[:, :, i2] = a * 2.0 ** -21 * nrm
    return t


def check_close(y, ref, dtype, extra=0.0):
    y = y.float().cpu().double().numpy()
    assert np.all(np.abs(y - ref) <= 1.5 * ulp(ref, dtype) + extra + 1e-7)


CASES = [
    # dense shape (B, L, H, d), rot_dim, interleaved, dtype
    ((2, 300, 3, 128), 128, False, torch.bfloat16),
    ((1, 1000, 2, 64), 64, True, torch.bfloat16),
    ((3, 77, 4, 128), 64, False, torch.float16),     # rotary on the first half of the features
    ((2, 33, 1, 64), 30, True, torch.bfloat16),     # rot_dim not a multiple of 8
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
@pytest.mark.parametrize("in_place", [False, True])
def test_rotary_dense(case, in_place):
    shape, rot, inter, dtype = case
    B, L, H, d = shape
    g = torch.Generator().manual_seed(sum(shape) + rot)
    x = torch.randn(*shape, generator=g).to(dtype)
    offs = torch.randint(0, 5000, (B,), generator=g, dtype=torch.int32)
    dev = torch.device("cuda", 0)
    xd = x.to(dev)
    y = attn.rotary(xd, rot, 10000.0, inter, offsets=offs.to(dev), out=xd if in_place else None)
    torch.cuda.synchronize()
    pos = (np.arange(L)[None, :] + offs.numpy()[:, None]).reshape(-1)
    ref = oracle.rotary(x.reshape(B * L, H, d), pos, rot, 10000.0, inter).reshape(B, L, H, d)
    extra = angle_term(x.reshape(B * L, H, d), pos, rot, inter).reshape(B, L, H, d)
    check_close(y, ref, dtype, extra)


def test_rotary_varlen_without_offsets():
    lengths = [5, 400, 1, 130]
    H, d = 2, 128
    g = torch.Generator().manual_seed(17)
    x = torch.randn(sum(lengths), H, d, generator=g).to(torch.bfloat16)
    cu = torch.tensor([0] + np.cumsum(lengths).tolist(), dtype=torch.int32)
    dev = torch.device("cuda", 0)
    y = attn.rotary(x.to(dev), cu_seqlens=cu.to(dev))
    torch.cuda.synchronize()
    pos = np.concatenate([np.arange(n) for n in lengths])
    check_close(y, oracle.rotary(x, pos, d), torch.bfloat16, angle_term(x, pos, d, False))


def test_rotary_then_cache_forward():
    # new tokens at positions cache_b .. cache_b + Lq_b - 1, keys at 0 .. Lk_b - 1
    lq, cache = [64, 200, 1, 37], [700, 33, 1999, 0]
    lk = [a + c for a, c in zip(lq, cache)]
    Hq, Hkv, d = 4, 2, 128
    g = torch.Generator().manual_seed(23)
    q = torch.randn(sum(lq), Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(sum(lk), Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(sum(lk), Hkv, d, generator=g).to(torch.bfloat16)
    cu_q = torch.tensor([0] + np.cumsum(lq).tolist(), dtype=torch.int32)
    cu_k = torch.tensor([0] + np.cumsum(lk).tolist(), dtype=torch.int32)
    dev = torch.device("cuda", 0)
    qr = attn.rotary(q.to(dev), cu_seqlens=cu_q.to(dev), offsets=torch.tensor(cache, dtype=torch.int32, device=dev))
    kr = attn.rotary(k.to(dev), cu_seqlens=cu_k.to(dev))
    o, lse = attn.attn_fwd(qr, kr, v.to(dev), causal=True, cu_seqlens=cu_q.to(dev), cu_seqlens_k=cu_k.to(dev))
    assert attn.get_error() == attn.ATTN_OK
    pos_q = np.concatenate([np.arange(n) + c for n, c in zip(lq, cache)])
    pos_k = np.concatenate([np.arange(n) for n in lk])
    # attn_rotary's output is the tensor's 16-bit type by contract: the
    # reference rounds its float64 rotation the same way before attention
    q_ref = torch.from_numpy(oracle.rotary(q, pos_q, d)).to(torch.bfloat16)
    k_ref = torch.from_numpy(oracle.rotary(k, pos_k, d)).to(torch.bfloat16)
    o_ref, lse_ref = oracle.varlen_cross_attention(q_ref, k_ref, v, lq, lk, causal=True, scale=d ** -0.5)
    o = o.float().cpu().double().numpy()
    assert float(np.abs(o - o_ref).max()) <= 1e-2
    assert float(np.abs(lse.cpu().double().numpy() - lse_ref).max()) <= 1e-3


def test_rotary_rejects_partial_overlap():
    dev = torch.device("cuda", 0)
    buf = torch.zeros(2 * 10 * 2 * 64 + 64, dtype=torch.bfloat16, device=dev)
    x = buf[:2 * 10 * 2 * 64].view(2, 10, 2, 64)
    y = buf[64:].view(2, 10, 2, 64)
    with pytest.raises(attn.AttnError):
        attn.rotary(x, out=y)


PACKED = [
    # (B, L, parts, H, d), rot_dim, interleaved, dtype, in_place
    ((2, 130, 3, 4, 128), 128, False, torch.bfloat16, True),    # qkv in place, as the module does
    ((1, 77, 3, 2, 64), 64, True, torch.float16, False),        # qkv out of place: v copied
    ((2, 50, 2, 3, 128), 64, False, torch.bfloat16, False),     # kv: only k rotated
    ((1, 40, 2, 2, 64), 30, False, torch.bfloat16, True),       # scalar path (rot_dim % 16 != 0)
]


@pytest.mark.parametrize("case", PACKED, ids=[f"packed{i}" for i in range(len(PACKED))])
def test_rotary_packed_qkv_and_kv(case):
    shape, rot, inter, dtype, in_place = case
    B, L, parts, H, d = shape
    g = torch.Generator().manual_seed(sum(shape) + rot)
    x = torch.randn(*shape, generator=g).to(dtype)
    offs = torch.randint(0, 3000, (B,), generator=g, dtype=torch.int32)
    dev = torch.device("cuda", 0)
    xd = x.to(dev)
    y = attn.rotary_packed(xd, rot, 10000.0, inter, offsets=offs.to(dev), out=xd if in_place else None)
    torch.cuda.synchronize()
    pos = (np.arange(L)[None, :] + offs.numpy()[:, None]).reshape(-1)
    y = y.cpu()
    for part in range(parts):
        xp = x[:, :, part].reshape(B * L, H, d)
        yp = y[:, :, part].reshape(B, L, H, d)
        if part == parts - 1:   # v: untouched, bit for bit
            assert torch.equal(yp, x[:, :, part])
            continue
        ref = oracle.rotary(xp, pos, rot, 10000.0, inter).reshape(B, L, H, d)
        check_close(yp, ref, dtype, angle_term(xp, pos, rot, inter).reshape(B, L, H, d))


def test_rotary_packed_varlen_qkv():
    lengths = [3, 200, 64]
    H, d = 2, 128
    g = torch.Generator().manual_seed(29)
    x = torch.randn(sum(lengths), 3, H, d, generator=g).to(torch.bfloat16)
    cu = torch.tensor([0] + np.cumsum(lengths).tolist(), dtype=torch.int32)
    dev = torch.device("cuda", 0)
    y = attn.rotary_packed(x.to(dev), cu_seqlens=cu.to(dev)).cpu()
    pos = np.concatenate([np.arange(n) for n in lengths])
    for part in range(2):
        check_close(y[:, part], oracle.rotary(x[:, part], pos, d), torch.bfloat16, angle_term(x[:, part], pos, d, False))
    assert torch.equal(y[:, 2], x[:, 2])
