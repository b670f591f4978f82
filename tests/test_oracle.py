"""Pins for the fp64 oracle, checked against things other than itself.

Every check here is independent of the oracle's own code: hand-worked values
(tests/golden/hand_worked.json), closed forms (delta filter = shifted input,
all-ones filter = box sums from an integral image, 1x1 = channel matmul,
output-size table), library routines that compute the same operation
(torch.nn.functional.conv2d in fp64 on the CPU, scipy.signal.correlate2d),
an explicit im2col-then-matmul written here, exact integer arithmetic, and
invariants (bias-only, linearity).  The mutation tests at the end plant
plausible mistakes in a copy of the oracle source and check that these pins
catch every one of them.
"""
import json
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch
import torch.nn.functional as F

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand(rng, *shape):
    return rng.standard_normal(size=shape)


def _torch_conv(x, w, b, stride, pad, dil):
    """Library routine: PyTorch's CPU conv2d in fp64 (NCHW / KCRS)."""
    y = F.conv2d(torch.from_numpy(x), torch.from_numpy(w),
                 None if b is None else torch.from_numpy(b),
                 stride=stride, padding=pad, dilation=dil)
    return y.numpy()


def _im2col_matmul(x, w, b, stride, pad, dil):
    """Explicit im2col then one matmul ("Output = Weight x im2col(Input)").

    Written independently of the oracle: pad the input, gather every window
    as one column with numpy slicing, multiply by the reshaped filters.
    """
    N, C, H, W = x.shape
    K, _, R, S = w.shape
    xp = np.pad(x, ((0, 0), (0, 0), (pad, pad), (pad, pad)))
    P = (H + 2 * pad - dil * (R - 1) - 1) // stride + 1
    Q = (W + 2 * pad - dil * (S - 1) - 1) // stride + 1
    cols = np.empty((N, C, R, S, P, Q))
    for r in range(R):
        for s in range(S):
            h0, w0 = r * dil, s * dil
            cols[:, :, r, s] = xp[:, :, h0:h0 + stride * (P - 1) + 1:stride,
                                  w0:w0 + stride * (Q - 1) + 1:stride]
    cols = cols.reshape(N, C * R * S, P * Q)
    y = np.einsum("kj,njm->nkm", w.reshape(K, C * R * S), cols).reshape(N, K, P, Q)
    if b is not None:
        y = y + b[None, :, None, None]
    return y


# ---------------------------------------------------------------- output size

SIZE_TABLE = [
    # (size, ksize, stride, pad, dil, expected) -- worked by hand
    (30, 3, 1, 1, 1, 30),   # MSCRED layer 1
    (30, 3, 2, 1, 1, 15),   # layer 2: floor(29/2)+1
    (15, 2, 2, 1, 1, 8),    # layer 3: floor(15/2)+1
    (8, 2, 2, 0, 1, 4),     # layer 4: floor(6/2)+1
    (56, 3, 1, 1, 1, 56),
    (28, 7, 1, 3, 1, 28),   # "same" padding
    (14, 3, 2, 1, 1, 7),
    (7, 1, 1, 0, 1, 7),
    (10, 3, 3, 0, 1, 3),    # floor(7/3)+1
    (5, 3, 1, 0, 2, 1),     # dilated window spans the whole input
    (5, 3, 1, 0, 3, 0),     # dilated window wider than the input: invalid
    (1, 1, 1, 0, 1, 1),
    (4, 5, 1, 0, 1, 0),
    (4, 5, 1, 1, 1, 2),
]


@pytest.mark.parametrize("size,k,st,pad,dil,expected", SIZE_TABLE)
def test_output_size_table(oracle_mod, size, k, st, pad, dil, expected):
    assert oracle_mod.out_extent(size, k, st, pad, dil) == expected


def test_output_size_matches_torch(oracle_mod):
    for size in range(1, 12):
        for k in range(1, 5):
            for st in (1, 2, 3):
                for pad in (0, 1, 2):
                    for dil in (1, 2):
                        got = oracle_mod.out_extent(size, k, st, pad, dil)
                        if size + 2 * pad - dil * (k - 1) - 1 < 0:
                            assert got == 0
                            continue
                        y = F.conv2d(torch.zeros(1, 1, size, 1), torch.zeros(1, 1, k, 1),
                                     stride=(st, 1), padding=(pad, 0), dilation=(dil, 1))
                        assert got == y.shape[2]


def test_mscred_chain_sizes(oracle_mod):
    h = 30
    for (k, st, pad), want in zip([(3, 1, 1), (3, 2, 1), (2, 2, 1), (2, 2, 0)], [30, 15, 8, 4]):
        h = oracle_mod.out_extent(h, k, st, pad, 1)
        assert h == want


# ---------------------------------------------------------------- hand-worked values

def test_hand_worked_golden(oracle_mod):
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x = np.array(c["x"], dtype=np.float64)
        w = np.array(c["w"], dtype=np.float64)
        b = None if c["bias"] is None else np.array(c["bias"], dtype=np.float64)
        y, _ = oracle_mod.conv2d(x, w, b, c["stride"], c["pad"], c["dil"])
        np.testing.assert_array_equal(y, np.array(c["y"], dtype=np.float64), err_msg=c["name"])


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("stride,pad,dil", [(1, 0, 1), (1, 2, 1), (2, 1, 1), (3, 2, 2), (1, 3, 3)])
def test_delta_filter_shifts_input(oracle_mod, stride, pad, dil):
    rng = np.random.default_rng(1)
    N, C, H, W, R, S = 2, 3, 9, 11, 3, 4
    x = _rand(rng, N, C, H, W)
    for r0 in range(R):
        for s0 in range(S):
            w = np.zeros((C, C, R, S))
            for k in range(C):
                w[k, k, r0, s0] = 1.0
            y, _ = oracle_mod.conv2d(x, w, None, stride, pad, dil)
            P, Q = y.shape[2:]
            exp = np.zeros_like(y)
            for p in range(P):
                for q in range(Q):
                    h = p * stride - pad + r0 * dil
                    ww = q * stride - pad + s0 * dil
                    if 0 <= h < H and 0 <= ww < W:
                        exp[:, :, p, q] = x[:, :, h, ww]
            np.testing.assert_array_equal(y, exp)


@pytest.mark.parametrize("R,S,pad", [(3, 3, 1), (5, 2, 0), (4, 4, 3), (1, 6, 2)])
def test_ones_filter_gives_box_sums(oracle_mod, R, S, pad):
    rng = np.random.default_rng(2)
    H, W = 13, 10
    x = rng.integers(-9, 10, size=(1, 1, H, W)).astype(np.float64)
    w = np.ones((1, 1, R, S))
    y, _ = oracle_mod.conv2d(x, w, None, 1, pad, 1)
    # integral image of the zero-padded input
    xp = np.pad(x[0, 0], pad)
    ii = np.zeros((xp.shape[0] + 1, xp.shape[1] + 1))
    ii[1:, 1:] = xp.cumsum(0).cumsum(1)
    P, Q = y.shape[2:]
    box = ii[R:R + P, S:S + Q] - ii[:P, S:S + Q] - ii[R:R + P, :Q] + ii[:P, :Q]
    np.testing.assert_array_equal(y[0, 0], box)


def test_1x1_is_channel_matmul(oracle_mod):
    rng = np.random.default_rng(3)
    x = _rand(rng, 3, 7, 5, 6)
    w = _rand(rng, 9, 7, 1, 1)
    b = _rand(rng, 9)
    y, _ = oracle_mod.conv2d(x, w, b, 1, 0, 1)
    exp = np.einsum("kc,nchw->nkhw", w[:, :, 0, 0], x) + b[None, :, None, None]
    np.testing.assert_allclose(y, exp, rtol=1e-13, atol=1e-13)


def test_bias_only(oracle_mod):
    rng = np.random.default_rng(4)
    x = _rand(rng, 2, 3, 6, 5)
    b = _rand(rng, 4)
    y, den = oracle_mod.conv2d(x, np.zeros((4, 3, 3, 3)), b, 2, 1, 1)
    np.testing.assert_array_equal(y, np.broadcast_to(b[None, :, None, None], y.shape))
    np.testing.assert_array_equal(den, np.broadcast_to(np.abs(b)[None, :, None, None], y.shape))


def test_linearity(oracle_mod):
    rng = np.random.default_rng(5)
    x1, x2 = _rand(rng, 2, 4, 8, 9), _rand(rng, 2, 4, 8, 9)
    w = _rand(rng, 5, 4, 3, 2)
    a = 0.75
    y12, _ = oracle_mod.conv2d(a * x1 + x2, w, None, 2, 1, 2)
    y1, _ = oracle_mod.conv2d(x1, w, None, 2, 1, 2)
    y2, _ = oracle_mod.conv2d(x2, w, None, 2, 1, 2)
    np.testing.assert_allclose(y12, a * y1 + y2, rtol=1e-12, atol=1e-12)


def test_scipy_correlate2d_single_channel(oracle_mod):
    from scipy.signal import correlate2d
    rng = np.random.default_rng(6)
    for pad in (0, 1, 2):
        x = _rand(rng, 1, 1, 12, 9)
        w = _rand(rng, 1, 1, 3, 4)
        y, _ = oracle_mod.conv2d(x, w, None, 1, pad, 1)
        exp = correlate2d(np.pad(x[0, 0], pad), w[0, 0], mode="valid")
        np.testing.assert_allclose(y[0, 0], exp, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- brute forces

def _random_shape(rng):
    while True:
        R, S = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        st, pad, dil = int(rng.integers(1, 4)), int(rng.integers(0, 4)), int(rng.integers(1, 4))
        H, W = int(rng.integers(1, 14)), int(rng.integers(1, 14))
        if H + 2 * pad - dil * (R - 1) - 1 >= 0 and W + 2 * pad - dil * (S - 1) - 1 >= 0:
            return (int(rng.integers(1, 4)), int(rng.integers(1, 6)), H, W,
                    int(rng.integers(1, 6)), R, S, st, pad, dil)


def test_against_im2col_matmul_and_torch(oracle_mod):
    rng = np.random.default_rng(7)
    for _ in range(60):
        N, C, H, W, K, R, S, st, pad, dil = _random_shape(rng)
        x, w = _rand(rng, N, C, H, W), _rand(rng, K, C, R, S)
        b = _rand(rng, K) if rng.integers(0, 2) else None
        y, den = oracle_mod.conv2d(x, w, b, st, pad, dil)
        e1 = _im2col_matmul(x, w, b, st, pad, dil)
        e2 = _torch_conv(x, w, b, st, pad, dil)
        scale = 1e-12 * max(1.0, float(np.abs(den).max()))
        np.testing.assert_allclose(y, e1, rtol=0, atol=scale)
        np.testing.assert_allclose(y, e2, rtol=0, atol=scale)
        # den is the same convolution applied to |x|, |w| plus |bias|
        ed = _torch_conv(np.abs(x), np.abs(w), None if b is None else np.abs(b), st, pad, dil)
        np.testing.assert_allclose(den, ed, rtol=0, atol=scale)


def test_exact_integer_arithmetic(oracle_mod):
    """Small integers: every partial sum is exact in fp64, so results match exactly."""
    rng = np.random.default_rng(8)
    for _ in range(30):
        N, C, H, W, K, R, S, st, pad, dil = _random_shape(rng)
        x = rng.integers(-8, 9, size=(N, C, H, W)).astype(np.float64)
        w = rng.integers(-8, 9, size=(K, C, R, S)).astype(np.float64)
        b = rng.integers(-8, 9, size=K).astype(np.float64)
        y, _ = oracle_mod.conv2d(x, w, b, st, pad, dil)
        np.testing.assert_array_equal(y, np.rint(_torch_conv(x, w, b, st, pad, dil)))


def test_nhwc_is_permuted_nchw(oracle_mod):
    rng = np.random.default_rng(9)
    x, w, b = _rand(rng, 2, 5, 7, 6), _rand(rng, 3, 5, 3, 2), _rand(rng, 3)
    y, den = oracle_mod.conv2d(x, w, b, 2, 1, 1)
    yh, denh = oracle_mod.conv2d(x.transpose(0, 2, 3, 1), w.transpose(0, 2, 3, 1), b, 2, 1, 1,
                                 layout="NHWC")
    np.testing.assert_array_equal(yh, y.transpose(0, 2, 3, 1))
    np.testing.assert_array_equal(denh, den.transpose(0, 2, 3, 1))


def test_points_equal_full(oracle_mod):
    rng = np.random.default_rng(10)
    x, w, b = _rand(rng, 3, 4, 9, 8), _rand(rng, 6, 4, 3, 3), _rand(rng, 6)
    y, den = oracle_mod.conv2d(x, w, b, 2, 1, 2)
    N, K, P, Q = y.shape
    idx = np.stack([rng.integers(0, d, size=50) for d in (N, K, P, Q)], axis=1)
    yp, dp = oracle_mod.conv2d_points(x, w, b, idx, 2, 1, 2)
    np.testing.assert_array_equal(yp, y[tuple(idx.T)])
    np.testing.assert_array_equal(dp, den[tuple(idx.T)])
    with pytest.raises(ValueError):
        oracle_mod.conv2d_points(x, w, b, [[0, 6, 0, 0]], 2, 1, 2)


def test_reduced_precision_inputs_read_exactly(oracle_mod):
    """bf16/fp16 inputs are widened exactly: same result as feeding the widened fp64 values."""
    rng = np.random.default_rng(11)
    for dt in (torch.float16, torch.bfloat16):
        x = torch.from_numpy(_rand(rng, 1, 3, 5, 5)).to(dt)
        w = torch.from_numpy(_rand(rng, 2, 3, 2, 2)).to(dt)
        y1, _ = oracle_mod.conv2d(x, w, None, 1, 1, 1)
        y2, _ = oracle_mod.conv2d(x.double().numpy(), w.double().numpy(), None, 1, 1, 1)
        np.testing.assert_array_equal(y1, y2)


def test_thread_count_does_not_change_result(oracle_mod):
    rng = np.random.default_rng(12)
    x, w, b = _rand(rng, 2, 6, 10, 10), _rand(rng, 8, 6, 3, 3), _rand(rng, 8)
    y1, _ = oracle_mod.conv2d(x, w, b, 1, 1, 1, threads=1)
    y4, _ = oracle_mod.conv2d(x, w, b, 1, 1, 1, threads=4)
    np.testing.assert_array_equal(y1, y4)


def test_error_ratio_semantics(oracle_mod):
    y_ref = np.array([1.0, 2.0, 0.0])
    den = np.array([2.0, 4.0, 0.0])
    assert oracle_mod.error_ratio(np.array([1.5, 2.0, 0.0]), y_ref, den) == pytest.approx(0.25)
    assert oracle_mod.error_ratio(np.array([1.0, 2.0, 1e-30]), y_ref, den) == float("inf")
    assert oracle_mod.error_ratio(np.array([np.nan, 2.0, 0.0]), y_ref, den) == float("inf")


# ---------------------------------------------------------------- planted mistakes

MUTATIONS = {
    "kernel_flip": ("int64_t h = p * stride - pad + r * dil;",
                    "int64_t h = p * stride - pad + (R - 1 - r) * dil;"),
    "pad_sign": ("int64_t ww = q * stride - pad + s * dil;",
                 "int64_t ww = q * stride + pad + s * dil;"),
    "dropped_bias": ("double acc = bias ? bias[k] : 0.0;", "double acc = 0.0;"),
    "h_bound_uses_W": ("if (h < 0 || h >= H) continue;", "if (h < 0 || h >= W) continue;"),
    "transposed_weight": ("double wv = w[((k * C + c) * R + r) * S + s];",
                          "double wv = w[((k * C + c) * S + s) * R + r];"),
    "stride_on_tap": ("int64_t h = p * stride - pad + r * dil;",
                      "int64_t h = p * stride - pad + r * stride;"),
    "size_off_by_one": ("return span / stride + 1;", "return (span + 1) / stride + 1;"),
    "den_signed": ("den += fabs(xv) * fabs(wv);", "den += xv * wv;"),
    "last_channel_dropped": ("for (int64_t c = 0; c < C; ++c) {", "for (int64_t c = 0; c + 1 < C; ++c) {"),
}


def _pins_pass(oracle_mod, lib):
    """A compact run of the pins above against another build; False on any failure."""
    rng = np.random.default_rng(13)
    try:
        for (size, k, st, pad, dil, exp) in SIZE_TABLE:
            if oracle_mod.out_extent(size, k, st, pad, dil, lib=lib) != exp:
                return False
        with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
            for c in json.load(f)["cases"]:
                b = None if c["bias"] is None else np.array(c["bias"], dtype=np.float64)
                y, _ = oracle_mod.conv2d(np.array(c["x"], dtype=np.float64),
                                         np.array(c["w"], dtype=np.float64), b,
                                         c["stride"], c["pad"], c["dil"], lib=lib)
                if not np.array_equal(y, np.array(c["y"], dtype=np.float64)):
                    return False
        for _ in range(20):
            N, C, H, W, K, R, S, st, pad, dil = _random_shape(rng)
            C = max(C, 2)
            x, w, b = _rand(rng, N, C, H, W), _rand(rng, K, C, R, S), _rand(rng, K)
            y, den = oracle_mod.conv2d(x, w, b, st, pad, dil, lib=lib)
            e = _torch_conv(x, w, b, st, pad, dil)
            ed = _torch_conv(np.abs(x), np.abs(w), np.abs(b), st, pad, dil)
            if y.shape != e.shape or not np.allclose(y, e, atol=1e-9) or not np.allclose(den, ed, atol=1e-9):
                return False
    except ValueError:
        return False
    return True


def test_pins_pass_on_the_real_oracle(oracle_mod):
    assert _pins_pass(oracle_mod, None)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(oracle_mod, name):
    src_path = os.path.join(os.path.dirname(HERE), "oracle", "conv2d_ref.c")
    src = open(src_path).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation anchor missing: {old}"
    with tempfile.TemporaryDirectory() as td:
        c_path = os.path.join(td, "mut.c")
        so_path = os.path.join(td, "mut.so")
        with open(c_path, "w") as f:
            f.write(src.replace(old, new, 1))
        subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
                        "-shared", c_path, "-o", so_path, "-lm"], check=True)
        lib = oracle_mod.load_build(so_path)
        assert not _pins_pass(oracle_mod, lib), f"planted mistake {name} went unnoticed"
