"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, none of which re-runs the oracle's own formula.

* the worked example 例 5-6 (S23-J17 §3.1): scores [0, ln 2], values [1, 3],
  one element per block -> r = 1/2, l' = 3/2, u' = 7/2, O = 7/3;
* rows of P sum to one, P >= 0 and masked keys get exactly zero weight;
* causal row 0 equals V[0] (the diagonal is the only allowed key);
* the blocked online recurrences of both pages equal the whole-row result by
  brute force on tiny inputs, for every block size;
* a library routine: torch's fp64 scaled_dot_product_attention on the CPU;
* closed forms: scale 0 gives the mean of V over the allowed keys and
  lse = ln |J_i|; one key gives V[0]; one dominant score gives its value row;
* structure: GQA equals MHA with K/V heads repeated; the padded batch with a
  key_padding_mask equals per-sequence runs; causal row i equals non-causal
  attention over the prefix 0..i; non-causal O is invariant under a joint
  permutation of the K/V rows;
* the byte accounting of the standard implementation (S23-J17 §3 table).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from tests.golden_fixtures import load

RNG = np.random.default_rng(20261202)


def rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# worked example
# ---------------------------------------------------------------------------

def _example_inputs(d=1):
    g = load("online_softmax_example_5_6.txt")
    # q = e0, k0 = 0, k1 = e0 and scale = ln 2 give the scores [0, ln 2]
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 2, 1, d))
    k[0, 1, 0, 0] = 1.0
    v = np.zeros((1, 2, 1, d))
    v[0, 0, 0, 0] = g["value_0"]
    v[0, 1, 0, 0] = g["value_1"]
    assert g["score_0"] == 0.0
    scale = g["score_1"]
    return g, q, k, v, scale


@pytest.mark.parametrize("d", [1, 64])
def test_worked_example_whole_row(d):
    g, q, k, v, scale = _example_inputs(d)
    o, lse = oracle.attention(q, k, v, scale=scale)
    assert abs(o[0, 0, 0, 0] - g["result"]) < 1e-15
    assert np.all(o[0, 0, 0, 1:] == 0.0)
    # lse = ln(e^0 + e^{ln 2}) = ln 3
    assert abs(lse[0, 0, 0] - math.log(3.0)) < 1e-15


@pytest.mark.parametrize("d", [1, 64])
def test_worked_example_online_trace(d):
    g, q, k, v, scale = _example_inputs(d)
    o, lse, tr = oracle.online_rows(q, k, v, [(0, 0, 0)], beta=1, form=0, scale=scale, trace=True)
    m0, l0, u0 = tr[0]
    m1, l1, u1 = tr[1]
    assert (m0, l0, u0) == (g["block_0_m"], g["block_0_l"], g["block_0_u"])
    assert abs(m1 - g["block_1_m"]) < 1e-15
    assert abs(l1 - g["block_1_l"]) < 1e-15
    assert abs(u1 - g["block_1_u"]) < 1e-15
    # the rescale factor is what turned l0 into l1 - 1 (the new block adds exp(0) = 1)
    assert abs((l1 - 1.0) / l0 - g["block_1_r"]) < 1e-15
    assert abs(o[0, 0] - g["result"]) < 1e-15
    # the normalised-o form reaches the same number
    o1, lse1, tr1 = oracle.online_rows(q, k, v, [(0, 0, 0)], beta=1, form=1, scale=scale, trace=True)
    assert abs(tr1[0][2] - 1.0) < 1e-15          # o after block 0 is v0
    assert abs(o1[0, 0] - g["result"]) < 1e-15
    assert abs(lse1[0] - math.log(3.0)) < 1e-15 and abs(lse[0] - math.log(3.0)) < 1e-15


# ---------------------------------------------------------------------------
# invariants of the definition
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(7, 7), (5, 9), (9, 5)])
def test_probability_rows_sum_to_one(causal, Lq, Lk):
    B, Hq, Hkv, d = 2, 4, 2, 8
    q, k, v = rand(B, Lq, Hq, d), rand(B, Lk, Hkv, d), rand(B, Lk, Hkv, d)
    o, lse, p = oracle.attention(q, k, v, causal=causal, with_probs=True)
    assert np.all(p >= 0.0)
    for i in range(Lq):
        allowed = [j for j in range(Lk) if (not causal) or j <= i + (Lk - Lq)]
        rows = p[:, :, i, :]
        if allowed:
            assert np.max(np.abs(rows.sum(-1) - 1.0)) < 1e-12
        else:
            assert np.all(rows == 0.0)
            assert np.all(o[:, i] == 0.0) and np.all(np.isneginf(lse[:, :, i]))
        masked = [j for j in range(Lk) if j not in allowed]
        assert np.all(rows[..., masked] == 0.0)


def test_padding_mask_rows_sum_to_one_and_skip_padding():
    B, L, H, d = 3, 6, 2, 4
    q, k, v = rand(B, L, H, d), rand(B, L, H, d), rand(B, L, H, d)
    mask = np.zeros((B, L), np.uint8)
    for b, n in enumerate([6, 3, 1]):
        mask[b, :n] = 1
    o, lse, p = oracle.attention(q, k, v, key_padding_mask=mask, with_probs=True)
    for b, n in enumerate([6, 3, 1]):
        assert np.max(np.abs(p[b, :, :n].sum(-1) - 1.0)) < 1e-12
        assert np.all(p[b, :, :, n:] == 0.0)
        # query rows that are padding produce nothing
        assert np.all(o[b, n:] == 0.0) and np.all(np.isneginf(lse[b, :, n:]))


def test_causal_row0_is_v0():
    B, L, Hq, Hkv, d = 2, 11, 4, 2, 16
    q, k, v = rand(B, L, Hq, d), rand(B, L, Hkv, d), rand(B, L, Hkv, d)
    scale = 0.37
    o, lse = oracle.attention(q, k, v, causal=True, scale=scale)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            assert np.array_equal(o[b, 0, h], v[b, 0, g])
            s00 = scale * float(np.dot(q[b, 0, h], k[b, 0, g]))
            assert abs(lse[b, h, 0] - s00) < 1e-13


# ---------------------------------------------------------------------------
# blocked online softmax == whole row, brute force on tiny inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("causal", [False, True])
def test_blocked_equals_whole_row(form, causal):
    rng = np.random.default_rng(7 + form + 2 * causal)
    for L in range(1, 10):
        for d in (1, 2, 4):
            q = rng.standard_normal((1, L, 2, d)) * 3.0
            k = rng.standard_normal((1, L, 1, d)) * 3.0
            v = rng.standard_normal((1, L, 1, d))
            rows = [(0, h, i) for h in range(2) for i in range(L)]
            o_ref, lse_ref = oracle.attention_rows(q, k, v, rows, causal=causal)
            for beta in range(1, L + 1):
                o, lse = oracle.online_rows(q, k, v, rows, beta=beta, form=form, causal=causal)
                assert np.max(np.abs(o - o_ref)) < 1e-12, (L, d, beta)
                assert np.max(np.abs(lse - lse_ref)) < 1e-12, (L, d, beta)


# ---------------------------------------------------------------------------
# a library routine: torch's fp64 SDPA on the CPU
# ---------------------------------------------------------------------------

def _torch_reference(q, k, v, causal, scale):
    """torch fp64 CPU attention through F.scaled_dot_product_attention; lse
    from torch.logsumexp of torch's own fp64 scores."""
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)          # B H L d
    kt = torch.from_numpy(k).permute(0, 2, 1, 3)
    vt = torch.from_numpy(v).permute(0, 2, 1, 3)
    G = qt.shape[1] // kt.shape[1]
    kt = kt.repeat_interleave(G, dim=1)
    vt = vt.repeat_interleave(G, dim=1)
    Lq, Lk = qt.shape[2], kt.shape[2]
    mask = None
    if causal:
        i = torch.arange(Lq)[:, None]
        j = torch.arange(Lk)[None, :]
        mask = j <= i + (Lk - Lq)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    s = (qt @ kt.transpose(-1, -2)) * scale
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 2, 64, 64, 32), (2, 8, 2, 33, 33, 16), (1, 4, 4, 17, 40, 8)])
def test_against_torch_sdpa_fp64(causal, shape):
    B, Hq, Hkv, Lq, Lk, d = shape
    q, k, v = rand(B, Lq, Hq, d), rand(B, Lk, Hkv, d), rand(B, Lk, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, causal=causal, scale=scale)
    o_t, lse_t = _torch_reference(q, k, v, causal, scale)
    assert np.max(np.abs(o - o_t)) < 1e-12
    assert np.max(np.abs(lse - lse_t)) < 1e-12


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_mean_of_allowed_values(causal):
    B, L, Hq, Hkv, d = 1, 9, 2, 1, 5
    q, k, v = rand(B, L, Hq, d), rand(B, L, Hkv, d), rand(B, L, Hkv, d)
    o, lse = oracle.attention(q, k, v, causal=causal, scale=0.0)
    for i in range(L):
        n = i + 1 if causal else L
        assert np.max(np.abs(o[0, i] - v[0, :n, 0].mean(axis=0))) < 1e-13
        assert np.max(np.abs(lse[0, :, i] - math.log(n))) < 1e-13


def test_single_key_gives_v0():
    q, k, v = rand(2, 6, 3, 4), rand(2, 1, 3, 4), rand(2, 1, 3, 4)
    o, lse = oracle.attention(q, k, v, scale=0.7)
    for i in range(6):
        assert np.array_equal(o[:, i], v[:, 0])
    assert np.allclose(lse, 0.7 * np.einsum("bihc,bhc->bhi", q, k[:, 0]), atol=1e-13, rtol=0)


def test_dominant_score_selects_its_value():
    L, d = 8, 4
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, L, 1, d))
    k[0, 5, 0, 0] = 1e3
    v = rand(1, L, 1, d)
    o, lse = oracle.attention(q, k, v, scale=1.0)
    assert np.max(np.abs(o[0, 0, 0] - v[0, 5, 0])) < 1e-300 + 1e-15
    assert abs(lse[0, 0, 0] - 1e3) < 1e-12


# ---------------------------------------------------------------------------
# structure
# ---------------------------------------------------------------------------

def test_gqa_equals_mha_with_repeated_kv():
    B, L, Hq, Hkv, d = 2, 13, 8, 2, 8
    q, k, v = rand(B, L, Hq, d), rand(B, L, Hkv, d), rand(B, L, Hkv, d)
    o, lse = oracle.attention(q, k, v, causal=True)
    G = Hq // Hkv
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    o2, lse2 = oracle.attention(q, kr, vr, causal=True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # heads 0..3 share KV head 0: a change to KV head 1 leaves them alone
    k2 = k.copy()
    k2[:, :, 1] += rand(B, L, d)       # a per-key change (a uniform shift would cancel)
    o3, _ = oracle.attention(q, k2, v, causal=True)
    assert np.array_equal(o3[:, :, :G], o[:, :, :G])
    assert not np.allclose(o3[:, :, G:], o[:, :, G:])


@pytest.mark.parametrize("causal", [False, True])
def test_padded_mask_equals_per_sequence_runs(causal):
    lengths = [5, 1, 9, 3]
    H, d = 3, 4
    total = sum(lengths)
    q, k, v = rand(total, H, d), rand(total, H, d), rand(total, H, d)
    o_packed, lse_packed = oracle.varlen_attention(q, k, v, lengths, causal=causal)
    off = 0
    for n in lengths:
        o1, lse1 = oracle.attention(q[None, off:off + n], k[None, off:off + n], v[None, off:off + n],
                                    causal=causal)
        assert np.max(np.abs(o_packed[off:off + n] - o1[0])) < 1e-13
        assert np.max(np.abs(lse_packed[:, off:off + n] - lse1[0])) < 1e-13
        off += n


def test_causal_row_equals_noncausal_prefix():
    L, H, d = 10, 2, 6
    q, k, v = rand(1, L, H, d), rand(1, L, H, d), rand(1, L, H, d)
    o, lse = oracle.attention(q, k, v, causal=True)
    for i in range(L):
        o1, lse1 = oracle.attention(q[:, i:i + 1], k[:, :i + 1], v[:, :i + 1], causal=False)
        assert np.max(np.abs(o[:, i] - o1[:, 0])) < 1e-13
        assert np.max(np.abs(lse[:, :, i] - lse1[:, :, 0])) < 1e-13


def test_noncausal_joint_permutation_invariance():
    L, H, d = 12, 2, 5
    q, k, v = rand(1, L, H, d), rand(1, L, H, d), rand(1, L, H, d)
    perm = RNG.permutation(L)
    o, lse = oracle.attention(q, k, v)
    o2, lse2 = oracle.attention(q, k[:, perm], v[:, perm])
    assert np.max(np.abs(o - o2)) < 1e-13 and np.max(np.abs(lse - lse2)) < 1e-13


def test_rows_routine_matches_full_routine_entries():
    B, L, Hq, Hkv, d = 2, 9, 4, 2, 8
    q, k, v = rand(B, L, Hq, d), rand(B, L, Hkv, d), rand(B, L, Hkv, d)
    o, lse = oracle.attention(q, k, v, causal=True)
    rows = [(1, 3, 8), (0, 0, 0), (1, 2, 4)]
    o_r, lse_r = oracle.attention_rows(q, k, v, rows, causal=True)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(o_r[n], o[b, i, h]) and lse_r[n] == lse[b, h, i]


def test_invalid_arguments_rejected():
    q, k, v = rand(1, 4, 3, 2), rand(1, 4, 2, 2), rand(1, 4, 2, 2)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v)          # 3 query heads over 2 KV heads


# ---------------------------------------------------------------------------
# byte accounting of the standard implementation
# ---------------------------------------------------------------------------

def test_standard_attention_traffic_table():
    g = load("standard_attention_traffic_l8192_d128.txt")
    t = oracle.standard_attention_traffic_bytes(int(g["L"]), int(g["d"]))
    assert t["q_each"] == g["q_each_bytes"]
    assert t["s"] == g["s_bytes"] and t["p"] == g["p_bytes"]
    assert t["qkvo"] == g["qkvo_bytes"]
    assert t["intermediate"] == g["intermediate_bytes"]
