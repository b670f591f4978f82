"""GPU parity of the MSCRED signature-matrix kernel against its fp64 oracle.

Tolerance, derived from the arithmetic: each entry is a fp32 FMA chain over
w products (each product exact inside the FMA, one rounding per step) and one
division by w, so |M - M_ref| <= (w + 1) * 2^-24 * den with
den = sum |s_i s_j| / w over the same samples; the tests allow (w_max + 2) * 2^-24.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import signature as sig_oracle
from cnn_convolution_gb300 import conv2d, workloads as wl
from parity import TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_convolution_gb300 import build
    build.build()
    conv2d.load()
    oracle.build()


def _check(series_cpu, windows, t_first, n_steps):
    out = conv2d.signature_matrices(series_cpu.cuda(), windows, t_first, n_steps)
    torch.cuda.synchronize()
    ref, den = sig_oracle.signature_matrices(series_cpu.numpy(), windows, t_first, n_steps)
    err = sig_oracle.error_ratio(out.cpu().numpy(), ref, den)
    tol = (max(windows) + 2) * 2.0 ** -24
    assert err <= tol, f"n={series_cpu.shape[0]} windows={windows}: err={err} > {tol}"
    return out


CASES = [
    # n_signals, T, windows, t_first, n_steps
    (1, 10, [1], 1, 10),
    (2, 5, [1, 2, 5], 5, 1),
    (5, 100, [30, 10, 60], 60, 41),          # unsorted windows
    (7, 200, [64, 65, 128, 3], 128, 73),     # odd signal count: a padded signal in the last blocks
    (30, 80, [10, 10, 30], 30, 51),          # a repeated window
    (40, 90, [17], 20, 70),                  # 210 pair blocks: padded to 224 per window
    (128, 50, [5, 50], 50, 1),               # the largest signal count: 2080 pair blocks per window
    (128, 120, [100, 3, 100], 100, 5),       # 52 KB of staged samples (above the default 48 KB)
    (20, 1400, [1300, 2], 1300, 7),          # too long to stage: read from global memory
    (128, 260, [7, 200], 200, 9),            # too long to stage at 128 signals
    (3, 64, [1, 2, 3, 4, 5, 6, 7, 8], 8, 57),   # eight windows, every length up to the history
]


@pytest.mark.parametrize("n,T,windows,t_first,n_steps", CASES)
def test_signature_matrices_parity(n, T, windows, t_first, n_steps):
    rng = np.random.default_rng(n * 1000 + T)
    s = torch.from_numpy(np.cumsum(rng.standard_normal((n, T)), axis=1).astype(np.float32))
    _check(s, windows, t_first, n_steps)


def test_mscred_encoder_input_on_gpu():
    """The encoder's layer-1 input, generated on the GPU from the raw signals."""
    s = wl.mscred_encoder_series(256)
    out = _check(s, list(wl.MSCRED_WINDOWS), 60, 256)
    assert tuple(out.shape) == (256, 3, 30, 30)


def test_signature_then_first_layer():
    """GPU signature matrices feed encoder layer 1 directly (NCHW, no copy)."""
    s = wl.mscred_encoder_series(32)
    x = conv2d.signature_matrices(s.cuda(), list(wl.MSCRED_WINDOWS), 60, 32)
    spec = wl.MSCRED_ENCODER[0]
    w, b = wl.mscred_encoder_params()[0]
    y = conv2d.forward(x, w.cuda(), b.cuda(), spec.stride, spec.pad, spec.dil, "NCHW")
    torch.cuda.synchronize()
    y_ref, den = oracle.conv2d(x.cpu(), w, b, spec.stride, spec.pad, spec.dil)
    assert oracle.error_ratio(y.cpu(), y_ref, den) <= TOL["f32"]


def test_signature_argument_errors():
    s = torch.zeros(4, 20, device="cuda")
    with pytest.raises(conv2d.Conv2dError):
        conv2d.signature_matrices(s, [10], 5, 1)          # window longer than the history
    with pytest.raises(conv2d.Conv2dError):
        conv2d.signature_matrices(s, [5], 10, 12)         # end times past the series
    with pytest.raises(conv2d.Conv2dError):
        conv2d.signature_matrices(s, [0], 10, 1)          # empty window
    assert conv2d.get_device_status() == 0
