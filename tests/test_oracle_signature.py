"""Pins of the signature-matrix oracle against what the definition fixes.

None of these re-types the oracle's loop: a hand-worked fixture, closed forms
(constant signals, a single sample, scaling), structure (symmetry, positive
semi-definiteness, nested windows adding up) and a planted-mistake check.
"""
import json
import os

import numpy as np
import pytest

from oracle import signature as sig

HERE = os.path.dirname(os.path.abspath(__file__))


def test_hand_worked_fixture():
    d = json.load(open(os.path.join(HERE, "golden", "signature_hand.json")))
    s = np.array(d["series"], dtype=np.float64)
    for case in d["cases"]:
        M, den = sig.signature_matrices(s, case["windows"], case["t_first"], case["n_steps"])
        np.testing.assert_allclose(M, np.array(case["M"]), rtol=0, atol=1e-15)
        assert np.all(den >= np.abs(M))


def test_constant_signals_give_outer_product():
    a = np.array([1.5, -2.0, 0.25])
    s = np.repeat(a[:, None], 40, axis=1)
    M, _ = sig.signature_matrices(s, [3, 10, 40], t_first=40, n_steps=1)
    for c in range(3):
        np.testing.assert_allclose(M[0, c], np.outer(a, a), rtol=1e-15)


def test_window_one_is_the_last_sample_outer_product():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((5, 12))
    M, _ = sig.signature_matrices(s, [1], t_first=4, n_steps=8)
    for b in range(8):
        col = s[:, 4 + b - 1]
        np.testing.assert_array_equal(M[b, 0], np.outer(col, col))


def test_symmetric_psd_and_scaling():
    rng = np.random.default_rng(4)
    s = np.cumsum(rng.standard_normal((6, 50)), axis=1)
    M, den = sig.signature_matrices(s, [5, 20], t_first=30, n_steps=4)
    assert np.array_equal(M, np.swapaxes(M, -1, -2))
    for m in M.reshape(-1, 6, 6):
        assert np.linalg.eigvalsh(m).min() > -1e-10 * np.abs(m).max()
    M2, _ = sig.signature_matrices(3.0 * s, [5, 20], t_first=30, n_steps=4)
    np.testing.assert_allclose(M2, 9.0 * M, rtol=1e-13)
    assert np.all(den >= np.abs(M) - 1e-12)


def test_nested_windows_add_up():
    # w2 * M(w2) = w1 * M(w1) + (w2 - w1) * M over the earlier samples only
    rng = np.random.default_rng(5)
    s = rng.standard_normal((4, 60))
    M, _ = sig.signature_matrices(s, [10, 30], t_first=50, n_steps=1)
    early, _ = sig.signature_matrices(s, [20], t_first=40, n_steps=1)
    np.testing.assert_allclose(30 * M[0, 1], 10 * M[0, 0] + 20 * early[0, 0], rtol=1e-12, atol=1e-12)


def test_matches_a_gram_matrix_of_the_window():
    rng = np.random.default_rng(6)
    s = rng.standard_normal((7, 25))
    M, _ = sig.signature_matrices(s, [9], t_first=20, n_steps=3)
    for b in range(3):
        seg = s[:, 20 + b - 9:20 + b]
        np.testing.assert_allclose(M[b, 0], seg @ seg.T / 9, rtol=1e-12, atol=1e-14)


def test_rejects_windows_outside_the_series():
    s = np.zeros((2, 10))
    with pytest.raises(ValueError):
        sig.signature_matrices(s, [5], t_first=4, n_steps=1)
    with pytest.raises(ValueError):
        sig.signature_matrices(s, [5], t_first=8, n_steps=4)


def test_error_ratio_flags_a_planted_mistake():
    # dividing by w - 1 instead of w (a plausible slip) is caught by the fixture scale
    rng = np.random.default_rng(7)
    s = rng.standard_normal((3, 30))
    M, den = sig.signature_matrices(s, [10], t_first=20, n_steps=2)
    assert sig.error_ratio(M, M, den) == 0.0
    assert sig.error_ratio(M * 10 / 9, M, den) > 1e-3
