"""Pins of the oracle's packed (varlen) backward, the per-sequence
composition of dense backwards (training page §2.5 packs sequences with
cumulative lengths; §5.3: the backward recomputes the weights).

The composition's own risk is its bookkeeping: the query and key offsets of
every sequence, empty sequences, and the bottom-right causal alignment of
sequences whose query and key lengths differ.  It is pinned by routes that
share none of that bookkeeping:

* torch autograd in fp64 through one attention over ALL packed rows with an
  explicit block-diagonal mask (same sequence, and for causal key j of a
  sequence visible to its query i iff j <= i + Lk_b - Lq_b), rows without a
  visible key contributing nothing;
* central finite differences of sum(dout * O) through the oracle's packed
  forward (varlen_cross_attention, pinned by brute force on its own);
* with equal query and key lengths, the dense backward of the padded batch
  with its key_padding_mask, scattered back to the packed rows.
"""

import numpy as np
import pytest
import torch

import oracle


def _masked_autograd(q, k, v, dout, lq, lk, causal, scale):
    """Gradients of sum(dout * O) for packed sequences through one masked
    attention over every packed row (block-diagonal mask)."""
    Tq, Hq, d = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    G = Hq // Hkv
    seq_q = np.repeat(np.arange(len(lq)), lq)
    seq_k = np.repeat(np.arange(len(lk)), lk)
    pos_q = np.concatenate([np.arange(n) for n in lq]) if Tq else np.zeros(0, int)
    pos_k = np.concatenate([np.arange(n) for n in lk]) if Tk else np.zeros(0, int)
    shift = np.asarray(lk)[seq_q] - np.asarray(lq)[seq_q] if Tq else np.zeros(0, int)
    allow = seq_q[:, None] == seq_k[None, :]
    if causal:
        allow &= pos_k[None, :] <= (pos_q + shift)[:, None]
    mask = torch.tensor(allow)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    Q = qt.permute(1, 0, 2)                                   # (Hq, Tq, d)
    K = kt.permute(1, 0, 2).repeat_interleave(G, 0)           # (Hq, Tk, d)
    V = vt.permute(1, 0, 2).repeat_interleave(G, 0)
    s = scale * Q @ K.transpose(1, 2)
    s = torch.where(mask[None], s, torch.tensor(-torch.inf, dtype=s.dtype))
    any_key = mask.any(dim=1)[None, :, None]
    m = torch.where(any_key, s.amax(dim=2, keepdim=True), torch.zeros(()).double())
    e = torch.where(mask[None], torch.exp(s - m), torch.zeros(()).double())
    p = e / torch.where(any_key, e.sum(dim=2, keepdim=True), torch.ones(()).double())
    o = (p @ V).permute(1, 0, 2)
    (o * torch.tensor(dout)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


CASES = [
    # query lengths, key lengths, Hq, Hkv, d
    ([3, 5, 4, 0, 2], [7, 5, 2, 3, 0], 4, 2, 5),     # longer, equal, shorter keys; empty pairings
    ([0, 6, 1], [4, 6, 1], 2, 1, 3),                  # empty query sequence first
    ([2, 2, 2], [5, 1, 3], 3, 3, 4),                  # causal rows with no key (Lq > Lk)
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c[0])))
def test_varlen_backward_matches_masked_autograd(case, causal):
    lq, lk, Hq, Hkv, d = case
    rng = np.random.default_rng(101 + 7 * len(lq) + int(causal))
    q = rng.standard_normal((sum(lq), Hq, d))
    k = rng.standard_normal((sum(lk), Hkv, d))
    v = rng.standard_normal((sum(lk), Hkv, d))
    dout = rng.standard_normal((sum(lq), Hq, d))
    got = oracle.varlen_attention_backward(q, k, v, dout, lq, lk, causal=causal, scale=0.6)
    ref = _masked_autograd(q, k, v, dout, lq, lk, causal, 0.6)
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert a.shape == b.shape, name
        assert np.allclose(a, b, atol=1e-11, rtol=0), f"{name}: {np.max(np.abs(a - b)):.3e}"


def test_varlen_backward_matches_finite_differences():
    lq, lk = [2, 0, 3], [3, 2, 2]
    Hq, Hkv, d, scale = 2, 1, 2, 0.8
    rng = np.random.default_rng(7)
    q = rng.standard_normal((sum(lq), Hq, d))
    k = rng.standard_normal((sum(lk), Hkv, d))
    v = rng.standard_normal((sum(lk), Hkv, d))
    dout = rng.standard_normal((sum(lq), Hq, d))
    got = oracle.varlen_attention_backward(q, k, v, dout, lq, lk, causal=True, scale=scale)

    def loss(xs):
        o, _ = oracle.varlen_cross_attention(xs[0], xs[1], xs[2], lq, lk, causal=True, scale=scale)
        return float(np.sum(o * dout))

    eps = 1e-5
    for which in range(3):
        xs = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(xs[which])
        for idx in np.ndindex(g.shape):
            x0 = xs[which][idx]
            xs[which][idx] = x0 + eps
            fp = loss(xs)
            xs[which][idx] = x0 - eps
            fm = loss(xs)
            xs[which][idx] = x0
            g[idx] = (fp - fm) / (2 * eps)
        assert np.allclose(got[which], g, atol=1e-7), f"input {which}: {np.max(np.abs(got[which] - g)):.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_equals_padded_route(causal):
    """Equal query and key lengths: the dense backward of the padded batch
    with a key_padding_mask, on the kept rows, is the packed result."""
    lens = [5, 1, 0, 8]
    Hq, Hkv, d = 4, 2, 3
    rng = np.random.default_rng(55 + int(causal))
    q = rng.standard_normal((sum(lens), Hq, d))
    k = rng.standard_normal((sum(lens), Hkv, d))
    v = rng.standard_normal((sum(lens), Hkv, d))
    dout = rng.standard_normal((sum(lens), Hq, d))
    got = oracle.varlen_attention_backward(q, k, v, dout, lens, lens, causal=causal, scale=0.5)
    qp, mask = oracle.pad_packed(q, lens)
    kp, _ = oracle.pad_packed(k, lens)
    vp, _ = oracle.pad_packed(v, lens)
    dp, _ = oracle.pad_packed(dout, lens)
    # padded query rows carry no loss: their dout is zero
    pq, pk, pv = oracle.attention_backward(qp, kp, vp, dp, causal=causal, scale=0.5, key_padding_mask=mask)
    keep = mask.astype(bool)
    for name, a, b in zip(("dq", "dk", "dv"), got, (pq[keep], pk[keep], pv[keep])):
        assert np.allclose(a, b, atol=1e-12), f"{name}: {np.max(np.abs(a - b)):.3e}"


def test_planted_offset_mistake_fails_the_pin():
    """A copy of the composition with one plausible bookkeeping mistake (the
    key offset advanced by the query length) must fail the masked route."""
    def buggy(q, k, v, dout, lq, lk, causal, scale):
        dq = np.zeros(q.shape)
        dk = np.zeros(k.shape)
        dv = np.zeros(k.shape)
        oq = ok = 0
        for nq, nk in zip(lq, lk):
            if nq > 0 and nk > 0:
                a, b_, c = oracle.attention_backward(q[None, oq:oq + nq], k[None, ok:ok + nk], v[None, ok:ok + nk],
                                                     dout[None, oq:oq + nq], causal=causal, scale=scale)
                dq[oq:oq + nq] = a[0]
                dk[ok:ok + nk] = b_[0]
                dv[ok:ok + nk] = c[0]
            oq += nq
            ok += nq      # planted: should advance by nk
        return dq, dk, dv

    lq, lk, Hq, Hkv, d = CASES[0]
    rng = np.random.default_rng(3)
    q = rng.standard_normal((sum(lq), Hq, d))
    k = rng.standard_normal((sum(lk), Hkv, d))
    v = rng.standard_normal((sum(lk), Hkv, d))
    dout = rng.standard_normal((sum(lq), Hq, d))
    got = buggy(q, k, v, dout, lq, lk, True, 0.6)
    ref = _masked_autograd(q, k, v, dout, lq, lk, True, 0.6)
    assert not all(np.allclose(a, b, atol=1e-11) for a, b in zip(got, ref))
