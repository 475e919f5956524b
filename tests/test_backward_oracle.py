"""Pins of the oracle's backward pass (gradients of sum(dout * O)).

The pages say only that the backward recomputes the attention weights from
what the forward kept (lei6393.com training-integration page, §5.3); the
gradients themselves follow from the forward's definition.  They are pinned
here by things other than their own formula:

* central finite differences of sum(dout * O) through the oracle's forward,
  which is pinned on its own (worked example, SDPA, closed forms);
* torch autograd through fp64 scaled_dot_product_attention (a library routine);
* invariants: the softmax gradient of a row sums to zero, so sum_j dk_j = 0,
  and the rows of P sum to one, so sum_j dv_j = sum_i dout_i;
* closed forms: one key (dq = dk = 0, dv = sum of dout), scale 0;
* padded keys get no gradient; the padded batch equals per-sequence runs.

A battery of these pins also runs against copies of the oracle with one
plausible mistake planted in the backward, each of which must fail a pin.
"""

import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle

SHAPES = [  # B, Hq, Hkv, Lq, Lk, d, causal
    (1, 2, 1, 5, 5, 3, False),
    (2, 4, 2, 6, 6, 4, True),
    (1, 2, 2, 4, 7, 3, True),     # causal, bottom-right aligned
    (1, 3, 1, 7, 4, 2, False),
]


def _rand(rng, B, Hq, Hkv, Lq, Lk, d):
    return (rng.standard_normal((B, Lq, Hq, d)), rng.standard_normal((B, Lk, Hkv, d)),
            rng.standard_normal((B, Lk, Hkv, d)), rng.standard_normal((B, Lq, Hq, d)))


def _fd(q, k, v, dout, causal, scale, L, eps=1e-5):
    """Central finite differences of sum(dout * O) with respect to q, k, v."""
    def loss(q_, k_, v_):
        o, _ = oracle.attention(q_, k_, v_, causal=causal, scale=scale, _lib=L)
        return float(np.sum(o * dout))

    grads = []
    for which in range(3):
        xs = [q.copy(), k.copy(), v.copy()]
        x = xs[which]
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + eps
            fp = loss(*xs)
            x[idx] = x0 - eps
            fm = loss(*xs)
            x[idx] = x0
            g[idx] = (fp - fm) / (2 * eps)
        grads.append(g)
    return grads


def _autograd(q, k, v, dout, causal, scale):
    B, Lq, Hq, d = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    Q = qt.permute(0, 2, 1, 3)
    K = kt.permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, 1)
    V = vt.permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, 1)
    mask = None
    if causal:
        mask = torch.arange(Lk)[None, :] <= torch.arange(Lq)[:, None] + (Lk - Lq)
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
    (o.permute(0, 2, 1, 3) * torch.tensor(dout)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def _battery(L):
    """Backward pins against oracle build ``L``; returns the failing names."""
    failed = []
    rng = np.random.default_rng(11)

    def check(name, cond):
        if not cond:
            failed.append(name)

    for shape in SHAPES:
        B, Hq, Hkv, Lq, Lk, d, causal = shape
        q, k, v, dout = _rand(rng, B, Hq, Hkv, Lq, Lk, d)
        sc = 1.0 / math.sqrt(d)
        dq, dk, dv = oracle.attention_backward(q, k, v, dout, causal=causal, scale=sc, _lib=L)
        fq, fk, fv = _fd(q, k, v, dout, causal, sc, L)
        check(f"finite_differences{shape}",
              max(np.abs(dq - fq).max(), np.abs(dk - fk).max(), np.abs(dv - fv).max()) < 1e-7)
        aq, ak, av = _autograd(q, k, v, dout, causal, sc)
        check(f"autograd{shape}",
              max(np.abs(dq - aq).max(), np.abs(dk - ak).max(), np.abs(dv - av).max()) < 1e-12)
        # invariants over the keys of each (batch, KV head); every query row
        # of these shapes has at least one allowed key
        G = Hq // Hkv
        sum_dout = dout.reshape(B, Lq, Hkv, G, d).sum(axis=(1, 3))
        check(f"sum_dk_zero{shape}", np.abs(dk.sum(axis=1)).max() < 1e-12)
        check(f"sum_dv{shape}", np.abs(dv.sum(axis=1) - sum_dout).max() < 1e-12)

    # one key: the weights are all one, nothing flows to q or k
    q, k, v, dout = _rand(rng, 1, 2, 1, 4, 1, 3)
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, _lib=L)
    check("one_key", np.abs(dq).max() == 0.0 and np.abs(dk).max() < 1e-14 and
          np.abs(dv[0, 0, 0] - dout[0].sum(axis=(0, 1))).max() < 1e-13)

    # scale 0: uniform weights over the allowed keys; dv_j = sum over the
    # rows that see key j of dout_i / |J_i|
    B, Hq, Hkv, L_, d = 1, 1, 1, 5, 3
    q, k, v, dout = _rand(rng, B, Hq, Hkv, L_, L_, d)
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, causal=True, scale=0.0, _lib=L)
    want = np.zeros((L_, d))
    for i in range(L_):
        want[:i + 1] += dout[0, i, 0] / (i + 1)
    check("zero_scale", np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0 and
          np.abs(dv[0, :, 0] - want).max() < 1e-13)

    # padded batch + mask: padded keys get nothing, kept rows match runs
    lengths = [3, 5]
    H, d = 2, 3
    tot = sum(lengths)
    q, k, v, dout = (rng.standard_normal((tot, H, d)) for _ in range(4))
    qp, mask = oracle.pad_packed(q, lengths)
    kp, _ = oracle.pad_packed(k, lengths)
    vp, _ = oracle.pad_packed(v, lengths)
    dp_, _ = oracle.pad_packed(dout, lengths)
    dq, dk, dv = oracle.attention_backward(qp, kp, vp, dp_, causal=True, key_padding_mask=mask, _lib=L)
    ok = np.abs(dk[0, 3:]).max() == 0.0 and np.abs(dv[0, 3:]).max() == 0.0
    off = 0
    for b, n in enumerate(lengths):
        r = oracle.attention_backward(q[None, off:off + n], k[None, off:off + n], v[None, off:off + n],
                                      dout[None, off:off + n], causal=True, _lib=L)
        ok &= max(np.abs(dq[b, :n] - r[0][0]).max(), np.abs(dk[b, :n] - r[1][0]).max(),
                  np.abs(dv[b, :n] - r[2][0]).max()) < 1e-13
        off += n
    check("padded_vs_runs", bool(ok))
    return failed


def test_backward_pins():
    assert _battery(oracle.lib()) == []


def test_backward_shapes_and_errors():
    rng = np.random.default_rng(1)
    q, k, v, dout = _rand(rng, 1, 2, 1, 3, 4, 2)
    dq, dk, dv = oracle.attention_backward(q, k, v, dout)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    with pytest.raises(ValueError):
        oracle.attention_backward(q, k, v, dout[:, :2])


MUTATIONS = {
    "drop_mean_dp": ("const double ds = prow[j] * (dp[j] - mean_dp);", "const double ds = prow[j] * dp[j];"),
    "ds_sign": ("const double ds = prow[j] * (dp[j] - mean_dp);", "const double ds = prow[j] * (mean_dp - dp[j]);"),
    "dq_without_scale": ("dq[qidx(b, i, h, c, Lq, Hq, d)] += scale * ds *", "dq[qidx(b, i, h, c, Lq, Hq, d)] += ds *"),
    "dk_from_keys": ("+= scale * ds * q[qidx(b, i, h, c, Lq, Hq, d)];", "+= scale * ds * k[kidx(b, j, g, c, Lk, Hkv, d)];"),
    "dv_without_p": ("+= prow[j] * dout[qidx(b, i, h, c, Lq, Hq, d)];", "+= dout[qidx(b, i, h, c, Lq, Hq, d)];"),
    "dp_against_keys": ("acc += dout[qidx(b, i, h, c, Lq, Hq, d)] * v[kidx(b, j, g, c, Lk, Hkv, d)];",
                        "acc += dout[qidx(b, i, h, c, Lq, Hq, d)] * k[kidx(b, j, g, c, Lk, Hkv, d)];"),
    "mean_unweighted": ("mean_dp += prow[j] * acc;", "mean_dp += acc;"),
    "gqa_one_head": ("for (int h = g * group; h < (g + 1) * group; ++h)", "for (int h = g * group; h < g * group + 1; ++h)"),
}


@pytest.fixture(scope="module")
def mutdir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_bwd_mut")


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_backward_mistake_is_caught(name, mutdir):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTATIONS[name]
    src = open(oracle.SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} is not unique in the oracle source"
    d = os.path.join(str(mutdir), name)
    os.makedirs(d, exist_ok=True)
    path_c = os.path.join(d, "oracle_mut.c")
    with open(path_c, "w", encoding="utf-8") as f:
        f.write(src.replace(old, new, 1))
    path_so = os.path.join(d, "liboracle_mut.so")
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", "-o", path_so, path_c, "-lm"],
                   check=True, capture_output=True)
    assert _battery(oracle.load_variant(path_so)), f"planted mistake {name} passed every pin"
