"""Parity of attn_bwd (dq, dk, dv) with the oracle's fp64 backward.

The forward runs on the GPU (attn_fwd) and its O and lse feed attn_bwd, as in
training; the oracle gets the same rounded q, k, v, dout and computes the
exact gradients of sum(dout * O) from the definition.

Bar, per gradient tensor X (derivation: the kernel rounds P and dS to the
input type before the tensor-core products, 2^-9 relative each for bf16,
forms D from the rounded O, and rounds X itself; every one of these is a
relative error of at most a few 2^-9 of the terms it touches, summed with
random signs):
    max |X - X_ref|  <= 2^-6 * max |X_ref|
    rms (X - X_ref)  <= 2^-7 * rms (X_ref)
A formula mistake (a missing D, scale, mask or head) moves X by O(|X|).
"""

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn

pytestmark = pytest.mark.gpu

MAX_TOL = 2.0 ** -6
RMS_TOL = 2.0 ** -7


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    return attn_lib


def make(B, Hq, Hkv, Lq, Lk, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Lq, Hq, d, generator=g).to(dtype)
    k = torch.randn(B, Lk, Hkv, d, generator=g).to(dtype)
    v = torch.randn(B, Lk, Hkv, d, generator=g).to(dtype)
    do = torch.randn(B, Lq, Hq, d, generator=g).to(dtype)
    return q, k, v, do


def gpu_grads(q, k, v, do, causal, scale):
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    assert attn.get_error() == attn.ATTN_OK
    return [t.float().cpu().double().numpy() for t in (dq, dk, dv)]


def check(name, x, ref):
    err = np.abs(x - ref)
    amax = float(np.abs(ref).max())
    rms_ref = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    assert np.all(np.isfinite(x)), name
    assert float(err.max()) <= MAX_TOL * amax + 1e-6, (name, float(err.max()), amax)
    assert float(np.sqrt(np.mean(err ** 2))) <= RMS_TOL * rms_ref + 1e-7, name


CASES = [
    # B, Hq, Hkv, Lq, Lk, d, causal, dtype
    (1, 2, 2, 256, 256, 64, False, torch.bfloat16),
    (1, 2, 1, 300, 300, 128, True, torch.bfloat16),      # GQA, ragged tail
    (2, 4, 2, 200, 333, 64, True, torch.float16),        # Lq != Lk, causal bottom-right
    (1, 1, 1, 130, 70, 128, True, torch.bfloat16),       # queries without keys (lse = -inf)
    (1, 2, 1, 1, 1, 64, False, torch.bfloat16),          # one query, one key
    (1, 4, 1, 513, 129, 128, False, torch.float16),
    (2, 2, 2, 640, 640, 128, True, torch.bfloat16),      # several tiles on both sides
    (1, 8, 1, 200, 200, 64, True, torch.bfloat16),       # eight query heads per KV head
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[:7]) for c in CASES])
def test_backward_matches_oracle(case):
    B, Hq, Hkv, Lq, Lk, d, causal, dtype = case
    q, k, v, do = make(B, Hq, Hkv, Lq, Lk, d, dtype, seed=sum(case[:6]))
    scale = d ** -0.5
    dq, dk, dv = gpu_grads(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, causal=causal, scale=scale)
    check("dq", dq, rq)
    check("dk", dk, rk)
    check("dv", dv, rv)
    if causal and Lq > Lk:
        # queries that see no key get no gradient
        blind = np.arange(Lq) + (Lk - Lq) < 0
        assert np.all(dq[:, blind] == 0.0)


def test_backward_zero_scale():
    # scale 0: uniform weights; dq and dk vanish, dv spreads dout evenly (a
    # closed form the oracle is pinned to)
    q, k, v, do = make(1, 2, 1, 150, 150, 128, torch.bfloat16, seed=8)
    dq, dk, dv = gpu_grads(q, k, v, do, False, 0.0)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, causal=False, scale=0.0)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0
    check("dv", dv, rv)


def test_backward_is_deterministic():
    q, k, v, do = make(1, 4, 2, 700, 700, 128, torch.bfloat16, seed=3)
    a = gpu_grads(q, k, v, do, True, 128 ** -0.5)
    b = gpu_grads(q, k, v, do, True, 128 ** -0.5)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_backward_empty_sides_give_zero():
    dev = torch.device("cuda", 0)
    for Lq, Lk in ((0, 64), (64, 0)):
        q, k, v, do = (t.to(dev) for t in make(1, 2, 1, Lq, Lk, 64, torch.bfloat16, seed=1))
        o = torch.zeros_like(q)
        lse = torch.full((1, 2, Lq), float("-inf"), device=dev)
        dq, dk, dv = (torch.full_like(t, 7.0) for t in (q, k, v))
        attn.attn_bwd(q, k, v, o, lse, do, causal=False, dq=dq, dk=dk, dv=dv)
        assert attn.get_error() == attn.ATTN_OK
        for t in (dq, dk, dv):
            assert torch.count_nonzero(t).item() == 0


def test_backward_full_size_group_sample():
    """The benchmark's backward workload (B2 Hq32 Hkv8 L4096 d128 causal):
    the whole problem runs on the GPU; the oracle evaluates one (batch, KV
    head) group, which is a self-contained sub-problem (its four query heads
    and its keys and values)."""
    B, Hq, Hkv, L, d = 2, 32, 8, 4096, 128
    q, k, v, do = make(B, Hq, Hkv, L, L, d, torch.bfloat16, seed=44)
    scale = d ** -0.5
    dq, dk, dv = gpu_grads(q, k, v, do, True, scale)
    G = Hq // Hkv
    b, g = 1, 5
    hs = slice(g * G, (g + 1) * G)
    rq, rk, rv = oracle.attention_backward(q[b:b + 1, :, hs], k[b:b + 1, :, g:g + 1], v[b:b + 1, :, g:g + 1],
                                           do[b:b + 1, :, hs], causal=True, scale=scale)
    check("dq", dq[b:b + 1, :, hs], rq)
    check("dk", dk[b:b + 1, :, g:g + 1], rk)
    check("dv", dv[b:b + 1, :, g:g + 1], rv)


def cu_of(lengths):
    return torch.tensor([0] + np.cumsum(lengths).tolist(), dtype=torch.int32)


VARLEN = [
    # query lengths, key lengths (None: self-attention, one offsets array), Hq, Hkv, d, causal, dtype
    ([37, 300, 1, 129], None, 4, 2, 64, True, torch.bfloat16),
    ([64, 200, 5, 256], [764, 233, 1005, 256], 4, 4, 128, True, torch.bfloat16),   # queries after a cache
    ([300, 20, 130], [100, 0, 130], 2, 1, 64, True, torch.float16),                 # keys < queries, no keys
    ([0, 17, 0, 400], [50, 3, 0, 300], 2, 2, 128, False, torch.bfloat16),          # empty sequences
    ([777], None, 2, 2, 64, True, torch.float16),                                   # one sequence
]


@pytest.mark.parametrize("case", VARLEN, ids=[f"varlen{i}" for i in range(len(VARLEN))])
def test_backward_varlen_matches_oracle(case):
    lq, lk, Hq, Hkv, d, causal, dtype = case
    self_attn = lk is None
    lk = lq if self_attn else lk
    g = torch.Generator().manual_seed(sum(lq) + sum(lk) + d)
    q = torch.randn(sum(lq), Hq, d, generator=g).to(dtype)
    k = torch.randn(max(sum(lk), 1), Hkv, d, generator=g).to(dtype)
    v = torch.randn(max(sum(lk), 1), Hkv, d, generator=g).to(dtype)
    do = torch.randn(sum(lq), Hq, d, generator=g).to(dtype)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    cq = cu_of(lq).to(dev)
    ck = None if self_attn else cu_of(lk).to(dev)
    scale = d ** -0.5
    o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, scale=scale, cu_seqlens=cq, cu_seqlens_k=ck)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, cu_seqlens=cq, cu_seqlens_k=ck)
    assert attn.get_error() == attn.ATTN_OK
    rq, rk, rv = oracle.varlen_attention_backward(q, k, v, do, lq, lk, causal=causal, scale=scale)
    nk = sum(lk)
    check("dq", dq.float().cpu().double().numpy(), rq)
    check("dk", dk.float().cpu().double().numpy()[:nk], rk[:nk])
    check("dv", dv.float().cpu().double().numpy()[:nk], rv[:nk])


def test_backward_varlen_equals_dense_for_equal_lengths():
    """Packed sequences of one length are the dense batch: the results agree
    bit for bit (the same kernels, the same tiles)."""
    B, L, Hq, Hkv, d = 3, 300, 4, 2, 128
    q, k, v, do = make(B, Hq, Hkv, L, L, d, torch.bfloat16, seed=9)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = attn.attn_fwd(qd, kd, vd, causal=True)
    a = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True)
    flat = lambda t: t.reshape(B * L, t.shape[2], d)
    lse_p = lse.permute(1, 0, 2).reshape(Hq, B * L).contiguous()
    cu = cu_of([L] * B).to(dev)
    b = attn.attn_bwd(flat(qd), flat(kd), flat(vd), flat(o), lse_p, flat(dod), causal=True, cu_seqlens=cu)
    assert attn.get_error() == attn.ATTN_OK
    for x, y in zip(a, b):
        assert torch.equal(flat(x), y)


def test_autograd_function_matches_oracle():
    """attn_func under torch.autograd: loss = sum(O * g) gives the oracle's
    gradients (dense, GQA, causal) and the forward's O."""
    B, Hq, Hkv, L, d = 1, 4, 2, 300, 64
    q, k, v, g = make(B, Hq, Hkv, L, L, d, torch.bfloat16, seed=12)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    o = attn.attn_func(qd, kd, vd, causal=True)
    (o.float() * g.to(dev).float()).sum().backward()
    assert attn.get_error() == attn.ATTN_OK
    rq, rk, rv = oracle.attention_backward(q, k, v, g, causal=True, scale=d ** -0.5)
    check("dq", qd.grad.float().cpu().double().numpy(), rq)
    check("dk", kd.grad.float().cpu().double().numpy(), rk)
    check("dv", vd.grad.float().cpu().double().numpy(), rv)
    o_ref, _ = oracle.attention(q, k, v, causal=True, scale=d ** -0.5)
    assert float(np.abs(o.detach().float().cpu().double().numpy() - o_ref).max()) <= 1e-2


def test_autograd_function_varlen():
    lengths = [50, 200, 7]
    Hq, Hkv, d = 2, 1, 128
    gen = torch.Generator().manual_seed(13)
    q = torch.randn(sum(lengths), Hq, d, generator=gen).to(torch.bfloat16)
    k = torch.randn(sum(lengths), Hkv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(sum(lengths), Hkv, d, generator=gen).to(torch.bfloat16)
    g = torch.randn(sum(lengths), Hq, d, generator=gen).to(torch.bfloat16)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    o = attn.attn_func(qd, kd, vd, causal=True, cu_seqlens=cu_of(lengths).to(dev))
    (o.float() * g.to(dev).float()).sum().backward()
    assert attn.get_error() == attn.ATTN_OK
    rq, rk, rv = oracle.varlen_attention_backward(q, k, v, g, lengths, lengths, causal=True, scale=d ** -0.5)
    check("dq", qd.grad.float().cpu().double().numpy(), rq)
    check("dk", kd.grad.float().cpu().double().numpy(), rk)
    check("dv", vd.grad.float().cpu().double().numpy(), rv)
