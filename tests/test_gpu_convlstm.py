"""GPU parity of the fused ConvLSTM cell (gate convolution on the 3xTF32
kernel, gates and state update in its epilogue) against the fp64 oracle.

Bounds (oracle/convlstm.py, ``tolerances``): each gate pre-activation may be
off by the fp32 convolution bound 1e-6 * den; sigmoid / tanh slopes carry it
into c and h; each fp32 activation or product adds at most 2^-21.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import N_TF_VARIANTS
from oracle import convlstm as lstm_oracle
from cnn_convolution_gb300 import conv2d, workloads as wl

pytestmark = pytest.mark.gpu
ACT_TOL = 2.0 ** -21


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_convolution_gb300 import build
    build.build()
    conv2d.load()
    oracle.build()


def _inputs(N, Cx, Ch, H, W, R, seed, bias=True):
    spec = wl.ConvSpec("cell", N, Cx + Ch, H, W, 4 * Ch, R, R, 1, R // 2, bias=bias)
    xh, w, b = wl.random_inputs(spec, seed=seed)
    rng = np.random.default_rng(seed + 7)
    c0 = torch.from_numpy(rng.uniform(-2, 2, size=(N, Ch, H, W)).astype(np.float32))
    return xh, w, b, c0


def _check(xh, w, b, c0, pad, c, h):
    c_ref, h_ref, _, den = lstm_oracle.cell(xh.numpy(), w.numpy(), None if b is None else b.numpy(),
                                            c0.numpy(), pad)
    dc, dh = lstm_oracle.tolerances(c0.numpy(), den, 1e-6, ACT_TOL)
    ec = np.abs(c.cpu().numpy().astype(np.float64) - c_ref)
    eh = np.abs(h.cpu().numpy().astype(np.float64) - h_ref)
    assert np.all(np.isfinite(ec)) and np.all(np.isfinite(eh))
    assert np.all(ec <= dc), f"c: worst excess {np.max(ec - dc)}"
    assert np.all(eh <= dh), f"h: worst excess {np.max(eh - dh)}"


CASES = [
    # N, Cx, Ch, H, W, R
    (2, 3, 4, 9, 11, 3),
    (1, 8, 8, 7, 7, 1),
    (3, 5, 7, 6, 13, 3),          # Ch not a multiple of any tile: ragged gate columns
    (2, 16, 16, 12, 12, 5),
    (2, 32, 32, 30, 30, 3),       # MSCRED layer-1 scale
    (4, 64, 64, 15, 15, 3),       # layer-2 scale
    (8, 128, 128, 8, 8, 3),       # layer-3 scale (gate conv K = 512)
    (4, 256, 256, 4, 4, 3),       # layer-4 scale: C*R*S = 4608, the 3-stage variant
]


@pytest.mark.parametrize("N,Cx,Ch,H,W,R", CASES)
def test_cell_parity(N, Cx, Ch, H, W, R):
    xh, w, b, c0 = _inputs(N, Cx, Ch, H, W, R, seed=N * 100 + Ch)
    c, h = conv2d.convlstm_cell(xh.cuda(), w.cuda(), b.cuda(), c0.cuda(), pad=R // 2)
    torch.cuda.synchronize()
    _check(xh, w, b, c0, R // 2, c, h)


def test_cell_without_bias_and_dilation():
    xh, w, _, c0 = _inputs(2, 6, 6, 10, 10, 3, seed=3, bias=False)
    c, h = conv2d.convlstm_cell(xh.cuda(), w.cuda(), None, c0.cuda(), pad=2, dil=2)
    torch.cuda.synchronize()
    c_ref, h_ref, _, den = lstm_oracle.cell(xh.numpy(), w.numpy(), None, c0.numpy(), 2, 2)
    dc, dh = lstm_oracle.tolerances(c0.numpy(), den, 1e-6, ACT_TOL)
    assert np.all(np.abs(c.cpu().numpy() - c_ref) <= dc)
    assert np.all(np.abs(h.cpu().numpy() - h_ref) <= dh)


def test_recurrence_writes_h_into_the_next_input():
    """Three steps; each step's h goes straight into the h slice of the next
    step's [x, h] buffer (h_img_stride = (Cx+Ch)*H*W)."""
    N, Cx, Ch, H, W = 2, 8, 8, 10, 10
    rng = np.random.default_rng(11)
    spec = wl.ConvSpec("cell", N, Cx + Ch, H, W, 4 * Ch, 3, 3, 1, 1)
    _, w, b = wl.random_inputs(spec, seed=12)
    xs = [torch.from_numpy(rng.standard_normal((N, Cx, H, W)).astype(np.float32)) for _ in range(3)]
    bufs = [torch.zeros(N, Cx + Ch, H, W, device="cuda") for _ in range(4)]
    c = torch.zeros(N, Ch, H, W, device="cuda")
    c_host, h_host = np.zeros((N, Ch, H, W)), np.zeros((N, Ch, H, W))
    for t in range(3):
        bufs[t][:, :Cx] = xs[t].cuda()
        nxt = bufs[t + 1]
        c, _ = conv2d.convlstm_cell(bufs[t], w.cuda(), b.cuda(), c, pad=1,
                                    h_next=nxt[:, Cx:], h_img_stride=(Cx + Ch) * H * W)
        torch.cuda.synchronize()
        # oracle step on exactly the state the GPU used (its own previous outputs)
        xh_used = bufs[t].cpu().numpy()
        c_ref, h_ref, _, den = lstm_oracle.cell(xh_used, w.numpy(), b.numpy(), c_host, 1)
        dc, dh = lstm_oracle.tolerances(c_host, den, 1e-6, ACT_TOL)
        got_h = nxt[:, Cx:].cpu().numpy()
        assert np.all(np.abs(c.cpu().numpy() - c_ref) <= dc)
        assert np.all(np.abs(got_h - h_ref) <= dh)
        c_host = c.cpu().numpy().astype(np.float64)
        h_host = got_h
    assert conv2d.get_device_status() == 0


def test_cell_argument_errors():
    xh = torch.zeros(1, 4, 6, 6, device="cuda")
    w = torch.zeros(8, 4, 3, 3, device="cuda")
    c0 = torch.zeros(1, 2, 6, 6, device="cuda")
    with pytest.raises(conv2d.Conv2dError):       # no padding: the map would shrink
        conv2d.convlstm_cell(xh, w, None, c0, pad=0)
    with pytest.raises(conv2d.Conv2dError):       # c_next aliasing c_prev
        conv2d.convlstm_cell(xh, w, None, c0, pad=1, c_next=c0)




@pytest.mark.parametrize("variant", range(N_TF_VARIANTS))
def test_cell_forced_variants(variant):
    """Every 3xTF32 variant that carries the gate epilogue (8 or more
    producer warps, one or two producer groups) gives the same cell; the
    others are refused as unsupported."""
    conv2d.set_override("tf_var", variant)
    try:
        ran = 0
        for i, (N, Cx, Ch, H, W, R) in enumerate([(2, 5, 7, 6, 13, 3), (2, 16, 16, 12, 12, 3)]):
            xh, w, b, c0 = _inputs(N, Cx, Ch, H, W, R, seed=500 + 10 * variant + i)
            try:
                c, h = conv2d.convlstm_cell(xh.cuda(), w.cuda(), b.cuda(), c0.cuda(), pad=R // 2)
            except conv2d.Conv2dError as e:
                assert e.code == 2, e
                continue
            torch.cuda.synchronize()
            _check(xh, w, b, c0, R // 2, c, h)
            ran += 1
    finally:
        conv2d.set_override("tf_var", None)
    if variant >= 3:    # 8 or more producer warps
        assert ran >= 1
