"""GPU parity of the transposed-convolution kernel against its fp64 oracle
(fp32 bound: max |y - y_ref| / (sum |x||w| + |bias|) <= 1e-6), including the
MSCRED decoder's four up-sampling shapes and edge geometry."""
import numpy as np
import pytest
import torch

import oracle
from oracle import deconv as dv_oracle
from cnn_convolution_gb300 import conv2d
from parity import N_TF_VARIANTS, TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_convolution_gb300 import build
    build.build()
    conv2d.load()
    oracle.build()


def _run(N, K, P, Q, C, R, S, st, pad, dil, op, bias=True, seed=0, dist="normal"):
    rng = np.random.default_rng(seed)
    if dist == "positive":
        x = rng.uniform(0, 1, (N, K, P, Q)); w = rng.uniform(0, 1, (K, C, R, S)); b = rng.uniform(0, 1, C)
    else:
        x = rng.standard_normal((N, K, P, Q))
        w = rng.standard_normal((K, C, R, S)) / np.sqrt(K * R * S)
        b = rng.uniform(-0.5, 0.5, C)
    x, w, b = (torch.from_numpy(a.astype(np.float32)) for a in (x, w, b))
    y = conv2d.deconv_forward(x.cuda(), w.cuda(), b.cuda() if bias else None, st, pad, dil, op)
    torch.cuda.synchronize()
    y_ref, den = dv_oracle.deconv2d(x.numpy(), w.numpy(), b.numpy() if bias else None, st, pad, dil, op)
    return oracle.error_ratio(y.cpu(), y_ref, den)


CASES = [
    # N, K, P, Q, C, R, S, stride, pad, dil, out_pad
    (2, 3, 5, 7, 4, 3, 3, 1, 1, 1, 0),
    (2, 8, 6, 6, 5, 3, 3, 2, 1, 1, 1),
    (1, 5, 9, 4, 3, 2, 2, 2, 0, 1, 0),       # kernel = stride: one tap per output
    (3, 4, 5, 5, 7, 5, 3, 3, 2, 1, 2),       # non-square filter, stride 3
    (2, 6, 7, 8, 33, 3, 3, 2, 1, 2, 1),      # dilation, 33 output channels: 2 channel blocks
    (1, 2, 1, 1, 3, 4, 4, 1, 0, 1, 0),       # one input pixel
    (2, 20, 11, 13, 9, 3, 3, 1, 0, 1, 0),    # output 13 x 15: ragged blocks
    (3, 11, 6, 9, 7, 2, 2, 1, 0, 1, 0),      # stride 1, 2x2, 8-channel block (one image per CTA)
    (2, 19, 4, 4, 8, 3, 3, 1, 2, 1, 0),      # stride 1, pad 2, ragged last input-channel chunk
    (1, 4, 70, 40, 3, 3, 3, 1, 1, 1, 0),     # stride 1, image too tall for one CTA: gather kernel
    # MSCRED decoder shapes (batch 8): 256->128 4->8, 256->64 8->15, 128->32 15->30, 64->3 30->30
    (8, 256, 4, 4, 128, 2, 2, 2, 0, 1, 0),
    (8, 256, 8, 8, 64, 3, 3, 2, 1, 1, 0),
    (8, 128, 15, 15, 32, 3, 3, 2, 1, 1, 1),
    (8, 64, 30, 30, 3, 3, 3, 1, 1, 1, 0),
]


@pytest.fixture(params=["tensor_core", "gather"])
def deconv_path(request):
    """The 3xTF32 tensor-core kernel per output residue class
    (CONV2D_DECONV_TC=1) and the gather kernel (CONV2D_DECONV_TC=0)."""
    with conv2d.overrides(deconv_tc=1 if request.param == "tensor_core" else 0):
        yield request.param


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_deconv_parity(case, deconv_path):
    err = _run(*case, seed=sum(case))
    assert err <= TOL["f32"], f"{case} ({deconv_path}): err={err}"


def test_deconv_class_without_taps_uses_the_gather_kernel():
    # stride 2 with a 1x1 filter: odd output rows receive no tap (bias only)
    assert _run(2, 4, 5, 5, 3, 1, 1, 2, 0, 1, 1, seed=11) <= TOL["f32"]


def test_deconv_without_bias_and_all_positive(deconv_path):
    assert _run(2, 16, 6, 6, 8, 3, 3, 2, 1, 1, 1, bias=False, seed=3) <= TOL["f32"]
    assert _run(2, 64, 8, 8, 16, 3, 3, 2, 1, 1, 0, seed=4, dist="positive") <= TOL["f32"]


def test_deconv_is_the_adjoint_on_the_gpu():
    """<conv(u), v> = <u, deconv(v)> with both sides computed by this library."""
    rng = np.random.default_rng(9)
    u = torch.from_numpy(rng.standard_normal((2, 6, 15, 15)).astype(np.float32)).cuda()
    w = torch.from_numpy(rng.standard_normal((8, 6, 3, 3)).astype(np.float32)).cuda()
    y = conv2d.forward(u, w, None, 2, 1, 1, "NCHW")                  # [2, 8, 8, 8]
    v = torch.from_numpy(rng.standard_normal(tuple(y.shape)).astype(np.float32)).cuda()
    z = conv2d.deconv_forward(v, w, None, 2, 1, 1, 0)                # [2, 6, 15, 15]
    lhs = float((y.double() * v.double()).sum())
    rhs = float((u.double() * z.double()).sum())
    scale = float((y.double() * v.double()).abs().sum())
    assert abs(lhs - rhs) <= 1e-5 * scale


def test_deconv_argument_errors():
    x = torch.zeros(1, 2, 3, 3, device="cuda")
    w = torch.zeros(2, 2, 3, 3, device="cuda")
    with pytest.raises(conv2d.Conv2dError):
        conv2d.deconv_forward(x, w, None, 2, 1, 1, 2)               # out_pad >= stride
    with pytest.raises(conv2d.Conv2dError):
        conv2d.deconv_forward(x.half(), w.half(), None, 1, 0)       # fp16: not supported
    assert conv2d.get_device_status() == 0


@pytest.mark.parametrize("variant", range(N_TF_VARIANTS))
def test_deconv_forced_variants(variant):
    """Each 3xTF32 variant in residue-class mode (a variant that cannot hold a
    class sends the layer to the gather kernel, which must agree too)."""
    with conv2d.overrides(tf_var=variant, deconv_tc=1):
        for case in [(2, 8, 6, 6, 5, 3, 3, 2, 1, 1, 1), (2, 6, 7, 8, 33, 3, 3, 2, 1, 2, 1),
                     (2, 20, 5, 5, 40, 2, 2, 2, 0, 1, 0)]:
            err = _run(*case, seed=900 + variant)
            assert err <= TOL["f32"], (case, variant, err)
