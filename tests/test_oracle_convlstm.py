"""Pins of the ConvLSTM-cell oracle against closed forms of the cell.

The gate convolution is the separately pinned convolution oracle; these
checks fix the gate order, the activations and the state update: zero
weights (gates = bias), saturated gates, a hand-worked 1x1 single-channel
step, and the recurrence identity with the forget gate open.
"""
import math

import numpy as np
import pytest

from oracle import convlstm


@pytest.fixture(scope="module", autouse=True)
def _built(oracle_mod):
    yield


def sig(z):
    return 1 / (1 + math.exp(-z))


def test_zero_weights_gates_are_the_bias():
    rng = np.random.default_rng(1)
    N, Cx, Ch, H, W = 2, 3, 2, 4, 5
    xh = rng.standard_normal((N, Cx + Ch, H, W))
    w = np.zeros((4 * Ch, Cx + Ch, 3, 3))
    b = np.array([0.5, -1.0, 2.0, 0.0, -0.25, 1.5, 0.3, -0.7])
    c0 = rng.standard_normal((N, Ch, H, W))
    c, h, _, _ = convlstm.cell(xh, w, b, c0, pad=1)
    for k in range(Ch):
        i, f, o, g = sig(b[k]), sig(b[Ch + k]), sig(b[2 * Ch + k]), math.tanh(b[3 * Ch + k])
        np.testing.assert_allclose(c[:, k], f * c0[:, k] + i * g, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(h[:, k], o * np.tanh(f * c0[:, k] + i * g), rtol=1e-13, atol=1e-15)


def test_saturated_gates():
    # i, o fully open, f fully closed: c = tanh(g_pre), h = tanh(c)
    rng = np.random.default_rng(2)
    xh = rng.standard_normal((1, 2, 3, 3))
    w = np.zeros((4, 2, 1, 1))
    w[3, 0, 0, 0] = 0.7                       # g = 0.7 * x channel 0
    b = np.array([60.0, -60.0, 60.0, 0.0])    # i, f, o pre-activations
    c0 = rng.standard_normal((1, 1, 3, 3))
    c, h, _, _ = convlstm.cell(xh, w, b, c0, pad=0)
    np.testing.assert_allclose(c[0, 0], np.tanh(0.7 * xh[0, 0]), rtol=1e-12, atol=1e-20)
    np.testing.assert_allclose(h[0, 0], np.tanh(np.tanh(0.7 * xh[0, 0])), rtol=1e-12)


def test_hand_worked_step():
    # 1x1 conv, Cx = Ch = 1, one pixel: x = 1, h = 2, c_prev = 0.5
    # z_i = 0.1*1 + 0.2*2 = 0.5; z_f = -0.3*1 + 0.1*2 = -0.1; z_o = 0.4*2 = 0.8; z_g = 1*1 - 0.5*2 = 0
    xh = np.array([[[[1.0]], [[2.0]]]])
    w = np.array([[0.1, 0.2], [-0.3, 0.1], [0.0, 0.4], [1.0, -0.5]]).reshape(4, 2, 1, 1)
    c, h, z, _ = convlstm.cell(xh, w, None, np.array([[[[0.5]]]]), pad=0)
    np.testing.assert_allclose(z.ravel(), [0.5, -0.1, 0.8, 0.0], atol=1e-15)
    c_exp = sig(-0.1) * 0.5 + sig(0.5) * 0.0
    assert abs(c[0, 0, 0, 0] - c_exp) < 1e-15
    assert abs(h[0, 0, 0, 0] - sig(0.8) * math.tanh(c_exp)) < 1e-15


def test_forget_gate_open_accumulates():
    # f = 1, i = 1, g = tanh(bias_g): c_t = c_{t-1} + tanh(b_g) step after step
    xh = np.zeros((1, 2, 2, 2))
    w = np.zeros((4, 2, 1, 1))
    b = np.array([60.0, 60.0, 0.0, 0.3])
    c = np.zeros((1, 1, 2, 2))
    for step in range(1, 4):
        c, h, _, _ = convlstm.cell(xh, w, b, c, pad=0)
        np.testing.assert_allclose(c, step * math.tanh(0.3), rtol=1e-12)


def test_shape_errors():
    with pytest.raises(ValueError):
        convlstm.cell(np.zeros((1, 2, 3, 3)), np.zeros((3, 2, 1, 1)), None, np.zeros((1, 1, 3, 3)), 0)
    with pytest.raises(ValueError):   # not "same": 3x3 without padding shrinks the map
        convlstm.cell(np.zeros((1, 2, 3, 3)), np.zeros((4, 2, 3, 3)), None, np.zeros((1, 1, 3, 3)), 0)
