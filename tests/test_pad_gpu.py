"""Parity of the padded-batch kernels (attn_unpad_index, row gather and
scatter, lse scatter) and of the padded forward built on them, through the C
ABI, with the oracle's plain definitions (lei6393.com training page, §2.5).

Index and row moves are exact: compared bit for bit.  The padded forward
meets the attention bar on kept rows (max |O - O_ref| <= 1e-2, max |lse -
lse_ref| <= 1e-3) and gives O = 0, lse = -inf at padded positions.
"""

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn
from tiled_attention_attn_gb300.inputs import WORKLOADS, generate

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    return attn_lib


def masks():
    g = torch.Generator().manual_seed(21)
    out = []
    lengths = [5, 130, 1, 256, 77]
    m = torch.zeros(len(lengths), 256, dtype=torch.bool)
    for b, n in enumerate(lengths):
        m[b, :n] = True
    out.append(("prefix", m))
    out.append(("holes", torch.rand(6, 300, generator=g) < 0.55))
    m = torch.rand(4, 1000, generator=g) < 0.3
    m[1] = False
    m[2] = True
    out.append(("empty and full rows", m))
    out.append(("one token", torch.ones(1, 1, dtype=torch.bool)))
    return out


@pytest.mark.parametrize("name,mask", masks(), ids=[n for n, _ in masks()])
def test_unpad_index_bitexact(name, mask):
    dev = torch.device("cuda", 0)
    cu, idx = attn.unpad_index(mask.to(dev))
    torch.cuda.synchronize()
    cu_ref, idx_ref = oracle.unpad_index(mask.numpy())
    assert cu.cpu().numpy().tolist() == cu_ref.tolist()
    total = int(cu_ref[-1])
    assert idx.cpu().numpy()[:total].tolist() == idx_ref.tolist()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_gather_scatter_bitexact(dtype):
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(3)
    B, L, H, d = 5, 300, 3, 64
    x = torch.randn(B, L, H, d, generator=g).to(dtype)
    mask = torch.rand(B, L, generator=g) < 0.6
    cu, idx = attn.unpad_index(mask.to(dev))
    n_dev = cu[B:]
    xd = x.to(dev)
    packed = attn.gather_rows(xd.view(B * L, H, d), idx, n_dev, B * L)
    cu_ref, idx_ref = oracle.unpad_index(mask.numpy())
    total = int(cu_ref[-1])
    ref = oracle.gather_rows(x.view(B * L, H, d).view(torch.int16).numpy(), idx_ref)
    assert np.array_equal(packed[:total].cpu().view(torch.int16).numpy(), ref)
    # back into a sentinel-filled padded buffer: kept rows restored, others untouched
    back = torch.full((B * L, H, d), 7.0, dtype=dtype, device=dev)
    attn.scatter_rows(packed, idx, n_dev, back)
    sentinel = int(torch.tensor(7.0, dtype=dtype).view(torch.int16).item())
    ref_back = oracle.scatter_rows(ref, idx_ref, B * L, fill=np.int16(sentinel))
    assert np.array_equal(back.cpu().view(torch.int16).numpy(), ref_back)


def test_row_count_comes_from_the_device():
    # the row count is read on the device; the gather zeroes the 128 rows
    # after it (the tile the attention kernels read past the last sequence)
    # and leaves the rows beyond those alone
    dev = torch.device("cuda", 0)
    src = torch.arange(300 * 8, dtype=torch.float32, device=dev).view(300, 8)
    idx = torch.arange(299, -1, -1, dtype=torch.int32, device=dev)
    n_dev = torch.tensor([10], dtype=torch.int32, device=dev)
    out = torch.full((300, 8), -1.0, device=dev)
    attn.gather_rows(src, idx, n_dev, 300, out=out)
    torch.cuda.synchronize()
    exp = torch.full((300, 8), -1.0)
    exp[:10] = src.cpu()[299 - torch.arange(10)]
    exp[10:138] = 0.0
    assert torch.equal(out.cpu(), exp)
    # an index outside the padded side moves nothing
    bad = torch.tensor([0, 70, -3, 5], dtype=torch.int32, device=dev)
    out2 = torch.full((64, 8), -1.0, device=dev)
    attn.scatter_rows(src[:4], bad, torch.tensor([4], dtype=torch.int32, device=dev), out2)
    exp2 = torch.full((64, 8), -1.0)
    exp2[0] = src.cpu()[0]
    exp2[5] = src.cpu()[3]
    assert torch.equal(out2.cpu(), exp2)


def test_scatter_lse_bitexact():
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(4)
    B, L, Hq = 3, 50, 5
    mask = torch.rand(B, L, generator=g) < 0.5
    cu, idx = attn.unpad_index(mask.to(dev))
    src = torch.randn(Hq, B * L, generator=g)
    out = torch.full((B, Hq, L), float("-inf"), device=dev)
    attn.scatter_lse(src.to(dev), idx, cu[B:], out)
    cu_ref, idx_ref = oracle.unpad_index(mask.numpy())
    ref = np.full((B, Hq, L), -np.inf, np.float32)
    for r, p in enumerate(idx_ref):
        b, i = divmod(int(p), L)
        ref[b, :, i] = src.numpy()[:, r]
    assert np.array_equal(out.cpu().numpy(), ref)


def check_padded(o, lse, o_ref, lse_ref, mask):
    m = mask.numpy()
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    assert np.all(o[~m] == 0.0)
    assert np.all(np.isneginf(lse.transpose(0, 2, 1)[~m]))
    assert float(np.abs(o[m] - o_ref[m]).max()) <= O_TOL
    lk = lse.transpose(0, 2, 1)[m]
    lk_ref = lse_ref.transpose(0, 2, 1)[m]
    fin = np.isfinite(lk_ref)
    assert np.array_equal(np.isfinite(lk), fin)
    assert float(np.abs(lk[fin] - lk_ref[fin]).max()) <= LSE_TOL


def test_padded_forward_varlen_config():
    # the varlen workload (B 16, H 12, d 64, lengths U[64, 512]) as a padded batch
    wl = WORKLOADS["varlen_b16_h12_d64"]
    inp = generate(wl)
    lengths = inp.lengths
    L = max(lengths)
    qp, mask = oracle.pad_packed(inp.q.float(), lengths, L)
    kp, _ = oracle.pad_packed(inp.k.float(), lengths, L)
    vp, _ = oracle.pad_packed(inp.v.float(), lengths, L)
    dev = torch.device("cuda", 0)
    dt = inp.q.dtype
    q = torch.from_numpy(qp).to(dt)
    k = torch.from_numpy(kp).to(dt)
    v = torch.from_numpy(vp).to(dt)
    maskt = torch.from_numpy(mask.astype(bool))
    o, lse = attn.attn_fwd_padded(q.to(dev), k.to(dev), v.to(dev), maskt.to(dev), causal=False)
    assert attn.get_error() == attn.ATTN_OK
    o_ref, lse_ref = oracle.padded_attention(q, k, v, mask, causal=False)
    check_padded(o, lse, o_ref, lse_ref, maskt)


@pytest.mark.parametrize("causal", [False, True])
def test_padded_forward_holes_gqa(causal):
    # kept tokens with holes (not a prefix), GQA 4:2, d 128
    g = torch.Generator().manual_seed(12 + int(causal))
    B, L, Hq, Hkv, d = 3, 300, 4, 2, 128
    mask = torch.rand(B, L, generator=g) < 0.7
    mask[2, :] = False
    q = torch.randn(B, L, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, L, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, L, Hkv, d, generator=g).to(torch.bfloat16)
    dev = torch.device("cuda", 0)
    o, lse = attn.attn_fwd_padded(q.to(dev), k.to(dev), v.to(dev), mask.to(dev), causal=causal)
    assert attn.get_error() == attn.ATTN_OK
    o_ref, lse_ref = oracle.padded_attention(q, k, v, mask.numpy(), causal=causal)
    check_padded(o, lse, o_ref, lse_ref, mask)


def test_padded_autograd_matches_oracle_with_poisoned_memory():
    """attn_func_padded forward and backward against the oracle's padded
    attention and backward (key-padding mask), after the caching allocator's
    memory was filled with NaN: the packed buffers past the kept rows must
    not leak into the results (the gather zeroes the tile past them)."""
    dev = torch.device("cuda", 0)
    poison = torch.full((64 << 20,), float("nan"), dtype=torch.float32, device=dev)
    del poison
    B, L, Hq, Hkv, d = 3, 200, 4, 2, 64
    g = torch.Generator().manual_seed(21)
    q = torch.randn(B, L, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, L, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, L, Hkv, d, generator=g).to(torch.bfloat16)
    go = torch.randn(B, L, Hq, d, generator=g).to(torch.bfloat16)
    lengths = [200, 131, 57]
    mask = torch.zeros(B, L, dtype=torch.bool)
    for b, n in enumerate(lengths):
        mask[b, :n] = True
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    o = attn.attn_func_padded(qd, kd, vd, mask.to(dev), causal=True)
    (o.float() * go.to(dev).float()).sum().backward()
    assert attn.get_error() == attn.ATTN_OK
    o_ref, _ = oracle.padded_attention(q, k, v, mask.numpy(), causal=True, scale=d ** -0.5)
    o_np = o.detach().float().cpu().double().numpy()
    assert np.all(np.isfinite(o_np)) and float(np.abs(o_np - o_ref).max()) <= 1e-2
    go_masked = go.clone()
    go_masked[~mask] = 0   # O is zero at padded positions, so they carry no gradient
    rq, rk, rv = oracle.attention_backward(q, k, v, go_masked, causal=True, scale=d ** -0.5,
                                           key_padding_mask=mask.numpy().astype(np.uint8))
    for name, x, r in (("dq", qd.grad, rq), ("dk", kd.grad, rk), ("dv", vd.grad, rv)):
        x = x.float().cpu().double().numpy()
        assert np.all(np.isfinite(x)), name
        assert float(np.abs(x - r).max()) <= 2.0 ** -6 * float(np.abs(r).max()) + 1e-6, name
        assert np.all(x[~mask.numpy()] == 0.0), name
