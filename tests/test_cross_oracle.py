"""Pins of the oracle's packed cross-attention / key-value-cache route
(training page §2.4, §4): brute force with explicit bottom-right masks, and
agreement with the padded self-attention route when the lengths match."""

import numpy as np
import pytest

import oracle


def _brute_cross(q, k, v, lq, lk, causal, scale):
    """Exact softmax attention of packed sequences written out row by row."""
    Hq, d = q.shape[1], q.shape[2]
    G = Hq // k.shape[1]
    o = np.zeros((q.shape[0], Hq, d))
    lse = np.full((Hq, q.shape[0]), -np.inf)
    oq = ok = 0
    for nq, nk in zip(lq, lk):
        for i in range(nq):
            for h in range(Hq):
                keys = [j for j in range(nk) if not causal or j <= i + nk - nq]
                if not keys:
                    continue
                s = np.array([scale * np.dot(q[oq + i, h], k[ok + j, h // G]) for j in keys])
                w = np.exp(s - s.max())
                o[oq + i, h] = sum(wj * v[ok + j, h // G] for wj, j in zip(w, keys)) / w.sum()
                lse[h, oq + i] = s.max() + np.log(w.sum())
        oq += nq
        ok += nk
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_cross_matches_brute_force(causal):
    # key lengths above, equal to and below the query lengths (rows with no key when causal)
    rng = np.random.default_rng(31 + int(causal))
    lq, lk = [3, 5, 4, 0, 2], [7, 5, 2, 3, 0]
    Hq, Hkv, d = 4, 2, 5
    q = rng.standard_normal((sum(lq), Hq, d))
    k = rng.standard_normal((sum(lk), Hkv, d))
    v = rng.standard_normal((sum(lk), Hkv, d))
    o, lse = oracle.varlen_cross_attention(q, k, v, lq, lk, causal=causal, scale=0.7)
    o_ref, lse_ref = _brute_cross(q, k, v, lq, lk, causal, 0.7)
    assert np.allclose(o, o_ref, atol=1e-12)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert np.allclose(lse[fin], lse_ref[fin], atol=1e-12)


def test_varlen_cross_equals_self_attention_route():
    # equal query and key lengths: the padded self-attention route must agree
    rng = np.random.default_rng(41)
    lens = [6, 1, 9]
    q = rng.standard_normal((sum(lens), 2, 8))
    k = rng.standard_normal((sum(lens), 2, 8))
    v = rng.standard_normal((sum(lens), 2, 8))
    for causal in (False, True):
        o1, l1 = oracle.varlen_cross_attention(q, k, v, lens, lens, causal=causal)
        o2, l2 = oracle.varlen_attention(q, k, v, lens, causal=causal)
        assert np.allclose(o1, o2, atol=1e-13) and np.allclose(l1, l2, atol=1e-13)
