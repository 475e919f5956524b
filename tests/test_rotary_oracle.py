"""Pins of the oracle's rotary embedding (training page §4).  The pages name
the knobs (rotary dimension, base, GPT-NeoX or GPT-J pairing, a position
offset) but print no formula; the reading is the standard rotation of each
feature pair by position * base^(-2p/rot_dim).  Pinned against complex
multiplication (numpy), and by the properties the embedding exists for."""

import numpy as np
import pytest

import oracle


def rng(seed):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotary_is_complex_multiplication(interleaved):
    r = rng(1 + int(interleaved))
    N, H, d, rot = 7, 3, 16, 12
    x = r.standard_normal((N, H, d))
    pos = r.integers(0, 5000, N)
    y = oracle.rotary(x, pos, rot, 10000.0, interleaved)
    half = rot // 2
    for p in range(half):
        i1, i2 = (2 * p, 2 * p + 1) if interleaved else (p, p + half)
        z = (x[:, :, i1] + 1j * x[:, :, i2]) * np.exp(1j * pos * 10000.0 ** (-2 * p / rot))[:, None]
        assert np.allclose(y[:, :, i1], z.real, atol=1e-12) and np.allclose(y[:, :, i2], z.imag, atol=1e-12)
    assert np.array_equal(y[:, :, rot:], x[:, :, rot:])


def test_rotary_position_zero_is_identity_and_additive():
    r = rng(3)
    x = r.standard_normal((5, 2, 8))
    assert np.array_equal(oracle.rotary(x, np.zeros(5), 8), x)
    p1, p2 = r.integers(0, 300, 5), r.integers(0, 300, 5)
    two = oracle.rotary(oracle.rotary(x, p1, 8), p2, 8)
    assert np.allclose(two, oracle.rotary(x, p1 + p2, 8), atol=1e-12)
    assert np.allclose(oracle.rotary(oracle.rotary(x, p1, 8), -p1, 8), x, atol=1e-12)


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotary_scores_depend_on_relative_position_only(interleaved):
    r = rng(7)
    d = 64
    q = r.standard_normal((1, 1, d))
    k = r.standard_normal((1, 1, d))
    dots = []
    for shift in (0, 17, 1000):
        qr = oracle.rotary(q, [40 + shift], d, 10000.0, interleaved)
        kr = oracle.rotary(k, [13 + shift], d, 10000.0, interleaved)
        dots.append(float(np.sum(qr * kr)))
    assert np.allclose(dots, dots[0], atol=1e-11)
    # and the norm of every pair is kept
    qr = oracle.rotary(q, [12345], d, 10000.0, interleaved)
    assert np.isclose(np.linalg.norm(qr), np.linalg.norm(q), atol=1e-12)


def test_gptj_is_neox_on_permuted_features():
    r = rng(9)
    N, H, d = 4, 2, 8
    x = r.standard_normal((N, H, d))
    pos = r.integers(0, 100, N)
    perm = np.array([0, 2, 4, 6, 1, 3, 5, 7])   # GPT-J pair (2p, 2p+1) -> GPT-NeoX pair (p, p+4)
    yj = oracle.rotary(x, pos, d, 10000.0, interleaved=True)
    yn = oracle.rotary(x[:, :, perm], pos, d, 10000.0, interleaved=False)
    assert np.allclose(yj[:, :, perm], yn, atol=1e-13)
