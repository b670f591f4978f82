"""GPU parity: the CUDA path against the fp64 oracle on seeded inputs.

Sizes span several tiles with ragged tails; every named workload runs at its
full size (sampled outputs where the whole output would take the oracle too
long), plus edge cases.  Tolerances are stated in tests/parity.py.
"""
import ctypes
import zlib

import numpy as np
import pytest
import torch

import oracle
from cnn_convolution_gb300 import conv2d, workloads as wl
from parity import TOL, full_parity, run_gpu, sampled_parity

pytestmark = pytest.mark.gpu

ALGOS_FOR = {
    ("f32", "NCHW"): ["auto"], ("f32", "NHWC"): ["auto"],
    ("f16", "NCHW"): ["auto"], ("bf16", "NCHW"): ["auto"],
    ("f16", "NHWC"): ["auto", "cuda_core"], ("bf16", "NHWC"): ["auto", "cuda_core"],
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_convolution_gb300 import build
    build.build()
    conv2d.load()
    oracle.build()


def _cases():
    for (dt, lay), algos in ALGOS_FOR.items():
        for algo in algos:
            yield dt, lay, algo


@pytest.mark.parametrize("dtype,layout,algo", list(_cases()))
def test_random_small_shapes(dtype, layout, algo):
    rng = np.random.default_rng(zlib.crc32(f"{dtype}{layout}{algo}".encode()))
    worst = 0.0
    for i in range(25):
        spec = wl.random_spec(rng, dtype, layout)
        if layout == "NHWC" and dtype != "f32" and i % 2 == 0:
            # channel counts the tensor-core path accepts (multiples of 8)
            spec = spec.replace(C=8 * int(rng.integers(1, 12)), K=8 * int(rng.integers(1, 12)))
        x, w, b = wl.random_inputs(spec, seed=1000 + i)
        err = full_parity(spec, x, w, b, algo)
        worst = max(worst, err)
        assert err <= TOL[dtype], f"{spec} err={err}"


RAGGED = [
    # M, K and C*R*S deliberately not multiples of any tile
    wl.ConvSpec("ragged_a", 3, 19, 23, 29, 71, 3, 3, 1, 1),
    wl.ConvSpec("ragged_b", 2, 40, 17, 31, 130, 2, 3, 2, 1),
    wl.ConvSpec("ragged_c", 5, 72, 13, 11, 200, 3, 3, 1, 2, 2),
    wl.ConvSpec("ragged_d", 1, 136, 33, 33, 264, 5, 5, 2, 2),
    wl.ConvSpec("ragged_e", 7, 64, 9, 9, 520, 1, 1, 1, 0),
    wl.ConvSpec("ragged_f", 2, 8, 40, 40, 24, 7, 7, 3, 3),
]


@pytest.mark.parametrize("dtype,layout", [("f32", "NCHW"), ("f32", "NHWC"), ("f16", "NHWC"),
                                          ("bf16", "NHWC"), ("bf16", "NCHW")])
@pytest.mark.parametrize("base", RAGGED, ids=lambda s: s.name)
def test_ragged_tiles(base, dtype, layout):
    spec = base.replace(dtype=dtype, layout=layout)
    x, w, b = wl.random_inputs(spec, seed=7)
    for algo in ALGOS_FOR[(dtype, layout)]:
        err = full_parity(spec, x, w, b, algo)
        assert err <= TOL[dtype], f"{algo}: err={err}"


EDGE = [
    wl.ConvSpec("one_pixel", 1, 1, 1, 1, 1, 1, 1),
    wl.ConvSpec("filter_wider_than_input", 2, 3, 3, 4, 5, 5, 5, 1, 2),
    wl.ConvSpec("single_output", 4, 16, 7, 7, 8, 7, 7, 1, 0),
    wl.ConvSpec("stride_gt_filter", 2, 8, 17, 19, 16, 2, 2, 5, 0),
    wl.ConvSpec("all_padding_taps", 1, 8, 2, 2, 8, 3, 3, 1, 3, bias=False),
    wl.ConvSpec("tall_thin", 1, 16, 97, 1, 16, 3, 1, 1, 1),
    wl.ConvSpec("dilated_3", 2, 16, 21, 21, 24, 3, 3, 2, 3, 3),
    wl.ConvSpec("asymmetric_filter", 2, 16, 12, 14, 16, 1, 5, 1, 2),
]


@pytest.mark.parametrize("dtype,layout", [("f32", "NCHW"), ("f32", "NHWC"), ("f16", "NHWC"),
                                          ("bf16", "NHWC")])
@pytest.mark.parametrize("spec", EDGE, ids=lambda s: s.name)
def test_edge_cases(spec, dtype, layout):
    spec = spec.replace(dtype=dtype, layout=layout)
    x, w, b = wl.random_inputs(spec, seed=11)
    for algo in ALGOS_FOR[(dtype, layout)]:
        err = full_parity(spec, x, w, b, algo)
        assert err <= TOL[dtype], f"{algo}: err={err}"


def test_all_padding_outputs_are_exact_zero():
    # pad 3 around a 2x2 image with a 3x3 filter: the corner outputs see only padding
    spec = wl.ConvSpec("pad_only", 1, 4, 2, 2, 4, 3, 3, 1, 3, bias=False)
    x, w, _ = wl.random_inputs(spec, seed=3)
    y, _ = run_gpu(spec, x, w, None)
    assert torch.all(y[:, :, 0, 0] == 0) and torch.all(y[:, :, -1, -1] == 0)


def test_long_reduction_rebuilds_tap_table():
    # C*R*S = 5400 > 4096 taps held in shared memory at once
    spec = wl.ConvSpec("long_reduction", 2, 600, 6, 6, 40, 3, 3, 1, 1)
    x, w, b = wl.random_inputs(spec, seed=5)
    assert full_parity(spec, x, w, b) <= TOL["f32"]


@pytest.mark.parametrize("C,R,st", [(64, 3, 1), (256, 3, 2), (128, 7, 1)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_all_positive_inputs(dtype, C, R, st):
    """Every product has the same sign: |y| = den, the hardest case for the
    bound (reductions of 576, 2304 and 6272 elements)."""
    spec = wl.ConvSpec("positive", 4, C, 14, 14, 64, R, R, st, R // 2, dtype=dtype, layout="NHWC")
    x, w, b = wl.random_inputs(spec, seed=9, dist="positive")
    for algo in ALGOS_FOR[(dtype, "NHWC")]:
        err = full_parity(spec, x, w, b, algo)
        print(f"all-positive {dtype} C*R*S={C * R * R} stride={st} {algo}: err={err:.3e}")
        assert err <= TOL[dtype], f"{algo}: err={err}"


# ------------------------------------------------------------ full-size workloads

def test_mscred_single_full():
    spec = wl.MSCRED_SINGLE
    x, w, b = wl.mscred_single_inputs()
    assert full_parity(spec, x, w, b) <= TOL["f32"]


@pytest.mark.parametrize("spec", wl.MSCRED_ENCODER, ids=lambda s: s.name)
def test_mscred_encoder_layer_full(spec):
    x, w, b = wl.workload_inputs(spec)
    assert full_parity(spec, x, w, b) <= TOL["f32"]


def test_mscred_encoder_chain():
    """The 4 layers chained on the signature-matrix batch; each layer is compared
    with the oracle applied to the input it actually received."""
    x = wl.mscred_encoder_input(256)
    params = wl.mscred_encoder_params()
    cur = x.cuda()
    for spec, (w, b) in zip(wl.MSCRED_ENCODER, params):
        y = conv2d.forward(cur, w.cuda(), b.cuda(), spec.stride, spec.pad, spec.dil, "NCHW")
        torch.cuda.synchronize()
        y_ref, den = oracle.conv2d(cur.cpu(), w, b, spec.stride, spec.pad, spec.dil)
        err = oracle.error_ratio(y.cpu(), y_ref, den)
        assert err <= TOL["f32"], f"{spec.name}: {err}"
        cur = y
    assert tuple(cur.shape) == (256, 256, 4, 4)


@pytest.mark.parametrize("spec", wl.TENSOR_CORE_WORKLOADS, ids=lambda s: s.name)
def test_tensor_core_workload_full_size(spec):
    x, w, b = wl.workload_inputs(spec)
    y, d = run_gpu(spec, x, w, b)
    assert d.workspace_bytes() == 0
    err = sampled_parity(spec, x, w, b, y)
    assert err <= TOL[spec.dtype], f"{d.plan()}: err={err}"
    assert torch.isfinite(y.float()).all()


# ------------------------------------------------------------ memory safety and streams

@pytest.mark.parametrize("dtype,layout", [("f32", "NCHW"), ("bf16", "NHWC"), ("f16", "NHWC")])
def test_guard_bands_untouched(dtype, layout):
    spec = wl.ConvSpec("guard", 3, 32, 15, 13, 40, 3, 3, 1, 1, dtype=dtype, layout=layout)
    x, w, b = wl.random_inputs(spec, seed=21)
    d = conv2d.Conv2dDesc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride,
                          spec.pad, spec.dil, spec.torch_dtype, spec.layout)
    shape = d.y_shape()
    n = int(np.prod(shape))
    guard = 4096
    buf = torch.full((n + 2 * guard,), float("nan"), dtype=spec.torch_dtype, device="cuda")
    y = buf[guard:guard + n].view(shape)
    d.forward(x.cuda(), w.cuda(), b.cuda(), y=y)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard].float()).all() and torch.isnan(buf[guard + n:].float()).all()
    y_ref, den = oracle.conv2d(x, w, b, spec.stride, spec.pad, spec.dil, layout=layout)
    assert oracle.error_ratio(y.cpu(), y_ref, den) <= TOL[dtype]


def test_side_stream_and_graph_capture():
    spec = wl.MSCRED_ENCODER[1].replace(N=8)
    x, w, b = wl.random_inputs(spec, seed=4)
    xd, wd, bd = x.cuda(), w.cuda(), b.cuda()
    d = conv2d.Conv2dDesc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride,
                          spec.pad, spec.dil)
    y_eager = d.forward(xd, wd, bd)
    s = torch.cuda.Stream()
    y_side = torch.empty_like(y_eager)
    with torch.cuda.stream(s):
        d.forward(xd, wd, bd, y=y_side)
    s.synchronize()
    y_graph = torch.empty_like(y_eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d.forward(xd, wd, bd, y=y_graph)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_eager, y_side) and torch.equal(y_eager, y_graph)


def test_host_pointers_rejected():
    lib = conv2d.load()
    x = torch.zeros(1, 3, 8, 8)          # CPU memory
    w = torch.zeros(4, 3, 3, 3)
    y = torch.zeros(1, 4, 8, 8)
    rc = lib.conv2d_forward(x.data_ptr(), w.data_ptr(), None, y.data_ptr(),
                            1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 0, 0, None)
    assert rc == 1
    xd = x.cuda()
    rc = lib.conv2d_forward(xd.data_ptr(), w.data_ptr(), None, y.data_ptr(),
                            1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 0, 0, None)
    assert rc == 1


def test_misaligned_device_pointer_rejected():
    lib = conv2d.load()
    buf = torch.zeros(4096, dtype=torch.float32, device="cuda")
    base = buf.data_ptr()
    rc = lib.conv2d_forward(ctypes.c_void_p(base + 2), ctypes.c_void_p(base + 1024), None,
                            ctypes.c_void_p(base + 8192), 1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 0, 0, None)
    assert rc == 3


def test_device_status_clean():
    assert conv2d.get_device_status() == 0


SPLIT_SHAPES = [
    wl.ConvSpec("split_a", 2, 64, 15, 15, 128, 2, 2, 2, 1),
    wl.ConvSpec("split_b", 3, 128, 8, 8, 256, 2, 2, 2, 0),
    wl.ConvSpec("split_c", 1, 37, 11, 13, 70, 3, 3, 1, 1),       # ragged everything
    wl.ConvSpec("split_d", 2, 600, 5, 5, 40, 3, 3, 1, 1),        # long reduction: tap-table rebuild
    wl.ConvSpec("split_e", 4, 96, 7, 9, 64, 3, 1, 2, 1, bias=False),
]


@pytest.mark.parametrize("layout", ["NCHW", "NHWC"])
@pytest.mark.parametrize("tile,split", [(0, 2), (1, 4), (2, 2), (6, 2), (6, 4), (7, 4)])
def test_cuda_core_split_k_clusters(tile, split, layout):
    """fp32 split-K: a cluster of `split` CTAs shares each output tile's
    reduction and sums the partial tiles through distributed shared memory."""
    with conv2d.overrides(cc_tile=tile, cc_split=split):
        for base in SPLIT_SHAPES:
            spec = base.replace(layout=layout)
            x, w, b = wl.random_inputs(spec, seed=31)
            y, d = run_gpu(spec, x, w, b, "cuda_core")
            assert f"split={split}" in d.plan(), d.plan()
            err = full_parity(spec, x, w, b, "cuda_core")
            assert err <= TOL["f32"], f"{spec.name} tile {tile} split {split}: {err}"
