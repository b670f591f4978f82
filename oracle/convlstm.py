"""Oracle for one ConvLSTM cell step: fp64 CPU.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

"GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch
Extension" (section "Understanding MSCRED": ConvLSTM keeps the spatial
structure of the encoded feature maps while it learns how they change over
time; its References cite the ConvLSTM paper of Shi et al., 2015).  The cell
taken here is that paper's, without the peephole terms (the plainest reading:
the page names no peepholes):

    z   = conv2d([x_t, h_{t-1}], W) + b          4*Ch channels, stride 1, "same"
    i   = sigmoid(z[0:Ch]),      f = sigmoid(z[Ch:2Ch]),
    o   = sigmoid(z[2Ch:3Ch]),   g = tanh(z[3Ch:4Ch])
    c_t = f * c_{t-1} + i * g
    h_t = o * tanh(c_t)

The gate convolution is the pinned convolution oracle (``oracle.conv2d``);
the rest is fp64 numpy elementwise math.  Returns the bounds the GPU result
is checked against as well (see ``tolerances``).
"""
from __future__ import annotations

import numpy as np

import oracle as _conv


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def cell(xh, w, bias, c_prev, pad: int, dil: int = 1):
    """One step.  xh: [N, Cx+Ch, H, W]; w: [4Ch, Cx+Ch, R, S] (gates i, f, o, g);
    bias: [4Ch] or None; c_prev: [N, Ch, H, W].  Returns (c, h, z, den), fp64;
    z are the gate pre-activations and den their conv error scales."""
    xh = np.asarray(xh, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    c_prev = np.asarray(c_prev, dtype=np.float64)
    N, C, H, W = xh.shape
    K = w.shape[0]
    if K % 4 or w.shape[1] != C:
        raise ValueError("w must be [4*Ch, Cx+Ch, R, S]")
    Ch = K // 4
    z, den = _conv.conv2d(xh, w, bias, 1, pad, dil, layout="NCHW")
    if z.shape[2:] != (H, W):
        raise ValueError("the gate convolution must keep H x W (same padding)")
    i = _sigmoid(z[:, 0:Ch])
    f = _sigmoid(z[:, Ch:2 * Ch])
    o = _sigmoid(z[:, 2 * Ch:3 * Ch])
    g = np.tanh(z[:, 3 * Ch:4 * Ch])
    c = f * c_prev + i * g
    h = o * np.tanh(c)
    return c, h, z, den


def tolerances(c_prev, den, conv_tol: float, act_tol: float):
    """Per-element bounds for c_t and h_t from a gate error bound.

    A pre-activation may be off by conv_tol * den (the convolution bound);
    sigmoid has slope <= 1/4 and tanh <= 1, and each activation or product in
    fp32 adds at most act_tol.  Then
      |dc| <= |c_prev| (dz_f / 4 + act_tol) + dz_i / 4 + dz_g + 3 act_tol
      |dh| <= dz_o / 4 + |dc| + 3 act_tol
    """
    c_prev = np.asarray(c_prev, dtype=np.float64)
    Ch = c_prev.shape[1]
    dz = conv_tol * den
    dz_i, dz_f, dz_o, dz_g = (dz[:, k * Ch:(k + 1) * Ch] for k in range(4))
    dc = np.abs(c_prev) * (dz_f / 4 + act_tol) + dz_i / 4 + dz_g + 3 * act_tol
    dh = dz_o / 4 + dc + 3 * act_tol
    return dc, dh
