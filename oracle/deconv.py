"""Oracle for the forward transposed convolution ("deconvolution"): fp64 CPU.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

"GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch
Extension" (section "Understanding MSCRED": the decoder reconstructs the
signature matrices from the encoded maps).  The decoder's up-sampling layer
is the transposed convolution: the adjoint of the forward convolution with
respect to its input.  Every input element x[n,k,p,q] spreads into the
output through the same taps the convolution would have gathered it from:

    y[n,c,h,w] = bias[c] + sum over k, p, q, r, s with
                 h = p*stride - pad + r*dil,  w = q*stride - pad + s*dil
                 of x[n,k,p,q] * wt[k,c,r,s]

x [N,K,P,Q], wt [K,C,R,S] (the forward conv's weights), y [N,C,H,W] with
H = (P-1)*stride - 2*pad + dil*(R-1) + 1 + out_pad (W likewise), out_pad in
[0, stride) choosing among the sizes whose forward convolution gives P.
"""
from __future__ import annotations

import numpy as np


def out_size(P: int, R: int, stride: int, pad: int, dil: int, out_pad: int = 0) -> int:
    return (P - 1) * stride - 2 * pad + dil * (R - 1) + 1 + out_pad


def deconv2d(x, wt, bias, stride: int, pad: int, dil: int = 1, out_pad: int = 0):
    """Return (y, den), fp64 NCHW; den = |bias| + sum of |x||wt| over the same terms."""
    x = np.asarray(x, dtype=np.float64)
    wt = np.asarray(wt, dtype=np.float64)
    N, K, P, Q = x.shape
    K2, C, R, S = wt.shape
    if K2 != K:
        raise ValueError("x and wt disagree on K")
    if not (0 <= out_pad < max(stride, dil)):
        raise ValueError("out_pad must be in [0, max(stride, dil))")
    H = out_size(P, R, stride, pad, dil, out_pad)
    W = out_size(Q, S, stride, pad, dil, out_pad)
    if H < 1 or W < 1:
        raise ValueError("empty output")
    y = np.zeros((N, C, H, W))
    den = np.zeros((N, C, H, W))
    ax, aw = np.abs(x), np.abs(wt)
    for p in range(P):
        for q in range(Q):
            for r in range(R):
                h = p * stride - pad + r * dil
                if not 0 <= h < H:
                    continue
                for s in range(S):
                    wc = q * stride - pad + s * dil
                    if not 0 <= wc < W:
                        continue
                    y[:, :, h, wc] += x[:, :, p, q] @ wt[:, :, r, s]
                    den[:, :, h, wc] += ax[:, :, p, q] @ aw[:, :, r, s]
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        y += b[None, :, None, None]
        den += np.abs(b)[None, :, None, None]
    return y, den
