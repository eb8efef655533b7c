"""Pins for the incoherent-processing oracle (oracle/incoherent.py).

Fixed by mathematics: the Sylvester construction of H_d (printed small cases,
H H^T = d I), the rotation M = diag(s) H_d / sqrt(d) is orthogonal, so
(Q M)(K M)^T = Q K^T ("FlashAttention-3 (BN)", section "Low precision (FP8)
and reducing quantisation error": the transform does not change Q K^T), and
the e4m3 round-trip bound of half an ulp (2^-4 relative for normal codes).
A planted mistake (a missing 1/sqrt(d)) is shown to break the invariance pin.
"""

import numpy as np

from oracle import incoherent
import synthetic


def test_small_hadamards_printed():
    assert np.array_equal(incoherent.hadamard(2), np.array([[1, 1], [1, -1]]))
    assert np.array_equal(incoherent.hadamard(4), np.array([[1, 1, 1, 1], [1, -1, 1, -1],
                                                            [1, 1, -1, -1], [1, -1, -1, 1]]))


def test_hadamard_orthogonality_and_rotation():
    for d in (64, 128):
        h = incoherent.hadamard(d)
        assert np.array_equal(h @ h.T, d * np.eye(d))
        m = incoherent.rotation(synthetic.random_signs(d, 3).numpy())
        assert np.abs(m @ m.T - np.eye(d)).max() < 1e-14


def test_scores_unchanged_by_rotation():
    r = np.random.default_rng(4)
    q, k = r.standard_normal((1, 9, 2, 128)), r.standard_normal((1, 11, 2, 128))
    s = synthetic.random_signs(128, 5).numpy()
    qr, kr = incoherent.rotate(q, s), incoherent.rotate(k, s)
    assert np.abs(np.einsum("bihd,bjhd->bhij", qr, kr) - np.einsum("bihd,bjhd->bhij", q, k)).max() < 1e-12
    # a rotation without the 1/sqrt(d) factor (a plausible slip) breaks it
    bad = q @ (s[:, None] * incoherent.hadamard(128))
    badk = k @ (s[:, None] * incoherent.hadamard(128))
    assert np.abs(np.einsum("bihd,bjhd->bhij", bad, badk) - np.einsum("bihd,bjhd->bhij", q, k)).max() > 1


def test_rotation_spreads_an_outlier():
    x = np.zeros((1, 1, 1, 128))
    x[0, 0, 0, 5] = 10.0
    y = incoherent.rotate(x, np.ones(128))
    assert np.allclose(np.abs(y), 10.0 / np.sqrt(128))


def test_quantiser_bounds():
    r = np.random.default_rng(6)
    y = r.standard_normal((2, 64, 3, 128)) * np.where(r.random((2, 64, 3, 128)) < 1e-3, 10, 1)
    codes, s = incoherent.quantize_e4m3_per_head(y)
    assert np.all(np.abs(codes).max(axis=(1, 3)) == 448.0)
    z = y / s.astype(np.float64)[:, None, :, None]
    err = np.abs(z - codes)
    normal = np.abs(z) >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(z[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * (1 + 1e-6))
