"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle
on the same seeded inputs, and compare with the tolerance of the method.

Tolerance (per output): |y_gpu - y_oracle| / (sum over taps of |x||w| + |bias|)
must not exceed 1e-6 for fp32 and 4e-3 for fp16 / bf16 inputs (fp32
accumulation, one round-to-nearest-even of the output).  Outputs whose taps
all fall in the padding with no bias must be exactly zero.
"""
import numpy as np
import torch

import oracle
from cnn_convolution_gb300 import conv2d, workloads as wl

TOL = {"f32": 1e-6, "f16": 4e-3, "bf16": 4e-3}

# Compiled 3xTF32 variants (the library's table).  Tests parametrize over
# range(N_TF_VARIANTS), and test_abi / test_gpu_fp32_tensor check that the
# library reports the same count, so a variant added there cannot go untested.
N_TF_VARIANTS = 17


def run_gpu(spec, x, w, b, algo="auto", stream=None):
    d = conv2d.Conv2dDesc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride,
                          spec.pad, spec.dil, spec.torch_dtype, spec.layout)
    if algo != "auto":
        d.set_algo(algo)
    xd, wd = x.cuda(), w.cuda()
    bd = None if b is None else b.cuda()
    y = d.forward(xd, wd, bd, stream=stream)
    torch.cuda.synchronize()
    return y.cpu(), d


def full_parity(spec, x, w, b, algo="auto"):
    """Whole-output comparison; returns the max error ratio."""
    y, _ = run_gpu(spec, x, w, b, algo)
    y_ref, den = oracle.conv2d(x, w, b, spec.stride, spec.pad, spec.dil, layout=spec.layout)
    assert tuple(y.shape) == y_ref.shape
    return oracle.error_ratio(y, y_ref, den)


def sampled_parity(spec, x, w, b, y, count=6000, seed=0, stratified=True):
    """Compare y (CPU tensor in spec.layout) at sampled logical outputs:
    random ones, the borders of the first and last image, and (stratified)
    points in every output tile."""
    if spec.layout == "NCHW":
        P, Q = y.shape[2], y.shape[3]
    else:
        P, Q = y.shape[1], y.shape[2]
    if stratified:
        idx = wl.check_points(spec, P, Q, seed, count)
    else:
        idx = wl.sample_indices(spec, P, Q, count, seed)
    y_ref, den = oracle.conv2d_points(x, w, b, idx, spec.stride, spec.pad, spec.dil,
                                      layout=spec.layout)
    n, k, p, q = idx.T
    got = y[n, k, p, q] if spec.layout == "NCHW" else y[n, p, q, k]
    return oracle.error_ratio(got, y_ref, den)
