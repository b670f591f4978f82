"""GPU parity of the direct fp32 kernel for short reductions (C*R*S <= 64).

Forced on (CONV2D_DIRECT=1) over both layouts: output blocks of 8 x 32
pixels with ragged edges in both directions, several 32-channel blocks and a
channel count that is not a multiple of 4 (scalar NHWC stores), strides,
padding wider than the filter, dilation, bias on and off, and the MSCRED
layers it serves (the single signature-matrix convolution and encoder layer 1).
"""
import os

import pytest
import torch

from cnn_convolution_gb300 import conv2d, workloads as wl
from parity import TOL, full_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_convolution_gb300 import build
    import oracle
    build.build()
    conv2d.load()
    oracle.build()


@pytest.fixture
def direct_on():
    with conv2d.overrides(direct=1):
        yield


SHAPES = [
    # N, C, H, W, K, R, S, stride, pad, dil, bias
    (2, 3, 30, 30, 32, 3, 3, 1, 1, 1, True),       # MSCRED layer 1 shape, small batch
    (1, 3, 40, 70, 70, 3, 3, 1, 1, 1, True),       # 3 column blocks, 3 channel blocks, ragged
    (2, 1, 9, 9, 5, 5, 5, 1, 2, 1, False),         # K % 4 != 0
    (3, 4, 33, 17, 16, 3, 3, 2, 1, 1, True),       # stride 2, ragged rows
    (1, 2, 20, 20, 8, 3, 3, 3, 4, 1, True),        # stride 3, pad wider than the filter
    (2, 7, 12, 12, 12, 3, 3, 1, 2, 2, True),       # dilation 2
    (1, 16, 10, 10, 40, 2, 2, 1, 0, 1, False),     # C*R*S = 64 exactly
    (2, 16, 6, 6, 8, 2, 2, 1, 0, 1, True),         # C*R*S = 64, K < one channel block
    (1, 1, 1, 1, 3, 1, 1, 1, 0, 1, True),          # one pixel
    (2, 5, 11, 13, 9, 3, 2, 1, 1, 1, True),        # non-square filter (generic tap loop)
    (1, 2, 23, 40, 33, 4, 4, 2, 3, 1, False),      # 4x4, stride 2, 33 channels
    # stride 1, dilation 1, K <= 32, 1x1 / 3x3 / 5x5: the register-blocked quad kernel
    (3, 3, 17, 45, 20, 3, 3, 1, 1, 1, True),       # K = 20: second channel half partly empty
    (2, 2, 9, 31, 7, 5, 5, 1, 2, 1, True),         # 5x5, Q not a multiple of 4
    (2, 5, 13, 14, 32, 1, 1, 1, 0, 1, False),      # 1x1
    (1, 6, 8, 33, 12, 3, 3, 1, 0, 1, True),        # no padding, a column block of 3
    (2, 2, 30, 30, 16, 5, 5, 1, 3, 1, True),       # pad wider than the filter half-width
]


@pytest.mark.parametrize("layout", ["NCHW", "NHWC"])
def test_direct_forced(layout, direct_on):
    for i, (N, C, H, W, K, R, S, st, pad, dil, bias) in enumerate(SHAPES):
        spec = wl.ConvSpec(f"dc{i}", N, C, H, W, K, R, S, st, pad, dil, layout=layout, bias=bias)
        x, w, b = wl.random_inputs(spec, seed=500 + i)
        y, d = run_gpu(spec, x, w, b, "cuda_core")
        assert "direct" in d.plan(), d.plan()
        err = full_parity(spec, x, w, b, algo="cuda_core")
        assert err <= TOL["f32"], f"{spec}: err={err}"


def test_direct_all_positive(direct_on):
    spec = wl.ConvSpec("dc_pos", 3, 7, 25, 37, 36, 3, 3, 1, 1)
    x, w, b = wl.random_inputs(spec, seed=7, dist="positive")
    assert full_parity(spec, x, w, b, algo="cuda_core") <= TOL["f32"]


def test_mscred_layers_direct(direct_on):
    spec = wl.MSCRED_SINGLE
    x, w, b = wl.mscred_single_inputs()
    assert full_parity(spec, x, w, b, algo="cuda_core") <= TOL["f32"]
    spec = wl.MSCRED_ENCODER[0]
    x, w, b = wl.workload_inputs(spec)
    y, d = run_gpu(spec, x, w, b, "cuda_core")
    assert "direct" in d.plan()
    assert full_parity(spec, x, w, b, algo="cuda_core") <= TOL["f32"]


def test_direct_not_used_where_it_cannot_apply(direct_on):
    # C*R*S = 72 > 64; and a stride-4 1x1 layer with 64 channels whose staged
    # patch (64 x 29 x 125 floats) exceeds the shared-memory budget
    for (C, R, st) in [(8, 3, 1), (64, 1, 4)]:
        d = conv2d.Conv2dDesc(2, C, 10, 10, 16, R, R, st, R // 2, 1, torch.float32, "NCHW")
        d.set_algo("cuda_core")
        assert "direct" not in d.plan(), d.plan()
