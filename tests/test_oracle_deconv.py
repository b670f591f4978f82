"""Pins of the transposed-convolution oracle.

The strongest: it is the adjoint of the (separately pinned) convolution
oracle, <conv(u), v> = <u, deconv(v)> for any u, v.  Plus closed forms
(stride 1 = convolution with the flipped, transposed filter; 1x1 = channel
matmul; kernel = stride spreads each input into its own block), the output
size against PyTorch, and PyTorch's own fp64 conv_transpose2d on random shapes.
"""
import numpy as np
import pytest
import torch

from oracle import deconv


@pytest.fixture(scope="module", autouse=True)
def _built(oracle_mod):
    yield


def _rand(rng, *shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("stride,pad,dil,R", [(1, 0, 1, 3), (2, 1, 1, 3), (2, 0, 1, 2), (3, 2, 2, 3), (2, 1, 2, 2)])
def test_adjoint_of_the_convolution(oracle_mod, stride, pad, dil, R):
    rng = np.random.default_rng(stride * 100 + pad * 10 + dil)
    N, C, K, H, W = 2, 3, 4, 11, 11
    wt = _rand(rng, K, C, R, R)
    u = _rand(rng, N, C, H, W)
    y, _ = oracle_mod.conv2d(u, wt, None, stride, pad, dil)             # [N, K, P, Q]
    P, Q = y.shape[2:]
    v = _rand(rng, N, K, P, Q)
    # choose out_pad so the transposed output has u's size
    op_h = H - deconv.out_size(P, R, stride, pad, dil)
    op_w = W - deconv.out_size(Q, R, stride, pad, dil)
    assert op_h == op_w and 0 <= op_h < max(stride, dil)
    z, _ = deconv.deconv2d(v, wt, None, stride, pad, dil, op_h)
    assert z.shape == u.shape
    assert abs(np.sum(y * v) - np.sum(u * z)) <= 1e-10 * np.sum(np.abs(y * v))


def test_stride_one_is_a_flipped_convolution(oracle_mod):
    rng = np.random.default_rng(2)
    x = _rand(rng, 2, 4, 6, 7)
    wt = _rand(rng, 4, 3, 3, 3)
    y, _ = deconv.deconv2d(x, wt, None, 1, 0)
    flipped = np.ascontiguousarray(wt[:, :, ::-1, ::-1].transpose(1, 0, 2, 3))
    z, _ = oracle_mod.conv2d(x, flipped, None, 1, 2, 1)
    np.testing.assert_allclose(y, z, rtol=1e-12, atol=1e-12)


def test_one_by_one_is_a_channel_matmul():
    rng = np.random.default_rng(3)
    x = _rand(rng, 2, 5, 4, 4)
    wt = _rand(rng, 5, 3, 1, 1)
    y, _ = deconv.deconv2d(x, wt, None, 1, 0)
    np.testing.assert_allclose(y, np.einsum("nkhw,kc->nchw", x, wt[:, :, 0, 0]), rtol=1e-13)


def test_kernel_equal_stride_places_blocks():
    rng = np.random.default_rng(4)
    x = _rand(rng, 1, 2, 3, 3)
    wt = _rand(rng, 2, 1, 2, 2)
    y, _ = deconv.deconv2d(x, wt, None, 2, 0)
    for p in range(3):
        for q in range(3):
            blk = np.einsum("k,krs->rs", x[0, :, p, q], wt[:, 0])
            np.testing.assert_allclose(y[0, 0, 2 * p:2 * p + 2, 2 * q:2 * q + 2], blk, rtol=1e-13)


def test_matches_torch_conv_transpose_fp64():
    rng = np.random.default_rng(5)
    for _ in range(20):
        st, dil = int(rng.integers(1, 4)), int(rng.integers(1, 3))
        R = int(rng.integers(1, 5))
        pad = int(rng.integers(0, 3))
        op = int(rng.integers(0, max(st, dil)))
        N, K, C = 2, int(rng.integers(1, 6)), int(rng.integers(1, 6))
        P, Q = int(rng.integers(1, 7)), int(rng.integers(1, 7))
        if deconv.out_size(P, R, st, pad, dil, op) < 1 or deconv.out_size(Q, R, st, pad, dil, op) < 1:
            continue
        x, wt, b = _rand(rng, N, K, P, Q), _rand(rng, K, C, R, R), _rand(rng, C)
        y, den = deconv.deconv2d(x, wt, b, st, pad, dil, op)
        ref = torch.nn.functional.conv_transpose2d(torch.from_numpy(x), torch.from_numpy(wt),
                                                   torch.from_numpy(b), stride=st, padding=pad,
                                                   output_padding=op, dilation=dil).numpy()
        np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)
        assert np.all(den >= np.abs(y) - 1e-12)
