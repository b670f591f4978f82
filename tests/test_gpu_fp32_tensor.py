"""GPU parity of the fp32 split-precision (3xTF32) tensor-core kernel, forced on.

Each fp32 operand is split into a TF32 high part and a TF32 low part and
every product is taken as hi*hi + hi*lo + lo*hi on the tensor cores.  The
result must meet the fp32 bound (1e-6 of sum |x||w| + |bias|) like the FFMA
kernel does; plain TF32 would miss it by two orders of magnitude.  Covers
both layouts, every compiled variant (tile width, pipeline depth, producer
warps), reductions that are not a multiple of the 32-element stage, ragged
M and K tiles, strides, padding, dilation, bias on and off, all-positive
inputs (every rounding error with the same sign) and the MSCRED encoder
layers at full size.
"""
import pytest
import torch

from cnn_convolution_gb300 import conv2d, workloads as wl
from parity import N_TF_VARIANTS, TOL, full_parity, run_gpu

pytestmark = pytest.mark.gpu

N_VARIANTS = N_TF_VARIANTS


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
def variant_env():
    def set_variant(v):
        conv2d.set_override("tf_var", v)
    yield set_variant
    conv2d.set_override("tf_var", None)


def test_variant_count_matches_library():
    assert conv2d.variant_count("tf32x3") == N_VARIANTS


SHAPES = [
    # N, C, H, W, K, R, S, stride, pad, dil, bias
    (1, 3, 30, 30, 32, 3, 3, 1, 1, 1, True),       # C*R*S = 27: one partial stage
    (2, 32, 15, 15, 64, 3, 3, 2, 1, 1, True),
    (3, 64, 8, 8, 128, 2, 2, 2, 1, 1, False),
    (2, 128, 4, 4, 256, 2, 2, 2, 0, 1, True),
    (2, 5, 11, 13, 7, 3, 3, 1, 1, 1, True),        # tiny C and K
    (1, 37, 9, 10, 70, 3, 2, 1, 2, 2, True),       # dilation, non-square filter, ragged K
    (3, 16, 17, 15, 40, 5, 5, 3, 2, 1, False),     # stride 3
    (2, 33, 7, 7, 264, 1, 1, 1, 0, 1, True),       # 1x1, ragged K past 256
    (1, 8, 3, 3, 16, 3, 3, 1, 0, 1, True),         # one output pixel per image
    (5, 24, 12, 12, 48, 3, 3, 1, 1, 1, True),      # several tiles per CTA
    (2, 5, 9, 11, 24, 2, 2, 1, 1, 2, True),        # 2x2 (table-free taps), dilation 2, C % 8 != 0
    (2, 13, 10, 7, 40, 2, 2, 2, 1, 1, False),      # 2x2 stride 2, ragged second stage
]


@pytest.mark.parametrize("layout", ["NCHW", "NHWC"])
@pytest.mark.parametrize("variant", range(N_VARIANTS))
def test_forced_variants(variant, layout, variant_env):
    variant_env(variant)
    ran = 0
    for i, (N, C, H, W, K, R, S, st, pad, dil, bias) in enumerate(SHAPES):
        spec = wl.ConvSpec(f"tf{i}", N, C, H, W, K, R, S, st, pad, dil, layout=layout, bias=bias)
        x, w, b = wl.random_inputs(spec, seed=300 + i)
        try:
            y, d = run_gpu(spec, x, w, b, "tensor_core")
        except conv2d.Conv2dError as e:
            # resident-weight variants need C*R*S small enough for every
            # stage's split weights to fit in shared memory
            assert e.code == 2, e
            continue
        assert "3xtf32" in d.plan(), d.plan()
        err = full_parity(spec, x, w, b, algo="tensor_core")
        assert err <= TOL["f32"], f"{spec} variant {variant}: err={err}"
        ran += 1
    assert ran >= 6


@pytest.mark.parametrize("layout", ["NCHW", "NHWC"])
@pytest.mark.parametrize("C,R", [(64, 3), (256, 3), (128, 5)])
def test_all_positive_long_reductions(C, R, layout):
    """x, w, bias ~ U(0, 1): |y| = den, and no rounding error cancels."""
    spec = wl.ConvSpec("tf_pos", 2, C, 9, 9, 64, R, R, 1, R // 2, layout=layout)
    x, w, b = wl.random_inputs(spec, seed=17, dist="positive")
    err = full_parity(spec, x, w, b, algo="tensor_core")
    print(f"all-positive C*R*S={C * R * R} {layout}: err={err:.3e}")
    assert err <= TOL["f32"], err


@pytest.mark.parametrize("spec", wl.MSCRED_ENCODER, ids=lambda s: s.name)
def test_mscred_encoder_layers(spec):
    x, w, b = wl.workload_inputs(spec)
    y, d = run_gpu(spec, x, w, b, "tensor_core")
    assert "3xtf32" in d.plan()
    err = full_parity(spec, x, w, b, algo="tensor_core")
    assert err <= TOL["f32"], f"{d.plan()}: err={err}"


def test_mscred_single():
    spec = wl.MSCRED_SINGLE
    x, w, b = wl.mscred_single_inputs()
    assert full_parity(spec, x, w, b, algo="tensor_core") <= TOL["f32"]


def test_deterministic_and_status_clean():
    spec = wl.ConvSpec("tf_det", 4, 32, 15, 15, 64, 3, 3, 2, 1)
    x, w, b = wl.random_inputs(spec, seed=8)
    y1, _ = run_gpu(spec, x, w, b, "tensor_core")
    y2, _ = run_gpu(spec, x, w, b, "tensor_core")
    assert torch.equal(y1, y2)
    assert conv2d.get_device_status() == 0
