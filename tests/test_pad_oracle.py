"""Pins of the oracle's unpad / pad definitions (lei6393.com training page,
§2.5): the page's padding example, equality with numpy's library routines
for arbitrary masks, and the round trip padded -> packed -> padded."""

import numpy as np
import pytest

import oracle
from tests.golden_fixtures import load


def test_unpad_index_training_page_example():
    g = load("unpad_training_page_2_5.txt")
    B, L, keep = int(g["B"]), int(g["L"]), int(g["kept_per_row"])
    mask = np.ones((B, L), bool)
    mask[:, keep:] = False
    cu, idx = oracle.unpad_index(mask)
    assert cu.tolist() == [int(g["cu_0"]), int(g["cu_1"]), int(g["cu_2"])]
    assert idx[int(g["cu_1"])] == int(g["first_index_row_1"])
    assert idx[-1] == int(g["last_index_row_1"])
    assert idx.tolist() == list(range(0, keep)) + list(range(L, L + keep))


@pytest.mark.parametrize("density", [0.0, 0.1, 0.5, 0.9, 1.0])
def test_unpad_index_matches_library_routines(density):
    rng = np.random.default_rng(int(density * 10) + 1)
    mask = rng.random((7, 33)) < density
    mask[3] = False            # a row with nothing kept
    mask[5] = True             # a row with everything kept
    cu, idx = oracle.unpad_index(mask)
    assert idx.tolist() == np.flatnonzero(mask).tolist()
    assert cu.tolist() == [0] + np.cumsum(mask.sum(axis=1)).tolist()


def test_gather_scatter_round_trip():
    rng = np.random.default_rng(5)
    B, L, H, d = 3, 17, 2, 8
    x = rng.standard_normal((B, L, H, d))
    mask = rng.random((B, L)) < 0.6
    cu, idx = oracle.unpad_index(mask)
    packed = oracle.gather_rows(x.reshape(B * L, H, d), idx)
    assert packed.shape == (int(cu[-1]), H, d)
    back = oracle.scatter_rows(packed, idx, B * L).reshape(B, L, H, d)
    assert np.array_equal(back, np.where(mask[:, :, None, None], x, 0.0))


def test_padded_attention_prefix_mask_equals_varlen():
    # a prefix mask is a varlen batch: both oracle routes must agree on the kept rows
    rng = np.random.default_rng(9)
    lengths = [5, 1, 9]
    L, H, d = max(lengths), 2, 8
    q = rng.standard_normal((sum(lengths), H, d))
    k = rng.standard_normal((sum(lengths), H, d))
    v = rng.standard_normal((sum(lengths), H, d))
    qp, mask = oracle.pad_packed(q, lengths, L)
    kp, _ = oracle.pad_packed(k, lengths, L)
    vp, _ = oracle.pad_packed(v, lengths, L)
    for causal in (False, True):
        o_pad, lse_pad = oracle.padded_attention(qp, kp, vp, mask, causal=causal)
        o_var, lse_var = oracle.varlen_attention(q, k, v, lengths, causal=causal)
        cu, idx = oracle.unpad_index(mask)
        assert np.allclose(oracle.gather_rows(o_pad.reshape(-1, H, d), idx), o_var, atol=1e-13)
        assert np.all(o_pad[mask == 0] == 0.0)
        assert np.all(np.isneginf(lse_pad.transpose(0, 2, 1)[mask == 0]))

