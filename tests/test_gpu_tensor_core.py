"""GPU parity of the tcgen05 / TMA-im2col tensor-core kernel, forced on.

Covers each output-channel tile width (64, 128, 256), channel counts that are
and are not multiples of the 64-channel k-block, output-channel counts that
leave a ragged tile, M not a multiple of 128 (tiles running past the last
image), strides, padding, dilation, non-square filters, bias on and off, and
several persistent rounds per CTA.
"""
import numpy as np
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
def force_bn():
    """Force a single-CTA im2col / plain variant (BN, KSUB)."""
    def set_bn(bn, ksub=None):
        conv2d.set_override("tc_bn", bn)
        conv2d.set_override("tc_ksub", ksub)
        conv2d.set_override("tc_cta2", 0)
    yield set_bn
    conv2d.set_override("tc_bn", None)
    conv2d.set_override("tc_ksub", None)
    conv2d.set_override("tc_cta2", None)


SHAPES = [
    # N, C, H, W, K, R, S, stride, pad, dil, bias
    (1, 64, 8, 8, 64, 3, 3, 1, 1, 1, True),
    (2, 64, 11, 13, 64, 3, 3, 1, 1, 1, False),
    (3, 128, 9, 7, 128, 3, 3, 2, 1, 1, True),
    (2, 8, 10, 10, 8, 3, 3, 1, 1, 1, True),        # C = K = 8: mostly zero-filled k-block
    (2, 72, 9, 9, 72, 3, 3, 1, 1, 1, True),        # C, K one past a multiple of 64
    (1, 200, 6, 6, 136, 2, 2, 1, 0, 1, False),
    (2, 64, 15, 15, 96, 5, 5, 1, 2, 1, True),
    (2, 32, 12, 14, 48, 1, 5, 1, 2, 1, True),      # non-square filter
    (2, 32, 14, 12, 48, 5, 1, 1, 2, 1, True),
    (2, 16, 13, 13, 40, 3, 3, 1, 2, 2, True),      # dilation 2
    (2, 24, 17, 15, 32, 3, 2, 3, 1, 1, True),      # stride 3
    (4, 64, 7, 7, 264, 1, 1, 1, 0, 1, True),       # 1x1, ragged K
    (5, 128, 14, 14, 256, 3, 3, 2, 1, 1, False),
    (1, 64, 3, 3, 64, 3, 3, 1, 0, 1, True),        # single output pixel per image
    (9, 64, 30, 30, 64, 3, 3, 1, 1, 1, True),      # many tiles: several persistent rounds
]


# (BN, k-blocks per pipeline stage): every compiled variant
VARIANTS = [(64, 2), (64, 4), (128, 1), (128, 2), (128, 3), (256, 1), (256, 2)]


@pytest.mark.parametrize("bn,ksub", VARIANTS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_forced_tile_widths(dtype, bn, ksub, force_bn):
    force_bn(bn, ksub)
    for i, (N, C, H, W, K, R, S, st, pad, dil, bias) in enumerate(SHAPES):
        spec = wl.ConvSpec(f"tc{i}", N, C, H, W, K, R, S, st, pad, dil, dtype=dtype,
                           layout="NHWC", bias=bias)
        x, w, b = wl.random_inputs(spec, seed=100 + i)
        err = full_parity(spec, x, w, b, algo="tensor_core")
        assert err <= TOL[dtype], f"{spec} BN={bn} KSUB={ksub}: err={err}"


def test_variant_counts_match_library():
    assert conv2d.variant_count("tensor_core") == len(VARIANTS)
    assert conv2d.variant_count("tensor_core_window") == len(WINDOW_VARIANTS)


# Persistent rounds: a CTA runs tiles blockIdx, blockIdx + grid, ...; the
# accumulator alternates between two tensor-memory buffers, the stage and
# accumulator phases flip every round and the epilogue's two staging buffers
# alternate.  A grid capped at a few CTAs makes each CTA run many rounds on a
# shape the oracle checks in full.
MULTI_ROUND_SHAPES = [
    # N, C, H, W, K, R, S, stride, pad, dil, bias
    (6, 64, 20, 20, 96, 3, 3, 1, 1, 1, True),      # 19 M tiles x 1-2 N tiles
    (4, 72, 17, 19, 136, 3, 3, 2, 1, 1, False),    # stride 2, ragged C, K and M
    (5, 128, 12, 12, 264, 1, 1, 1, 0, 1, True),    # 1x1 plain A, ragged K
]


@pytest.mark.parametrize("grid_cap", [1, 3])
@pytest.mark.parametrize("bn,ksub", VARIANTS)
def test_forced_variants_many_rounds_per_cta(bn, ksub, grid_cap, force_bn):
    force_bn(bn, ksub)
    with conv2d.overrides(grid_cap=grid_cap, tc_window=0):
        for i, (N, C, H, W, K, R, S, st, pad, dil, bias) in enumerate(MULTI_ROUND_SHAPES):
            spec = wl.ConvSpec(f"rounds{i}", N, C, H, W, K, R, S, st, pad, dil, dtype="bf16",
                               layout="NHWC", bias=bias)
            x, w, b = wl.random_inputs(spec, seed=700 + i)
            y, d = run_gpu(spec, x, w, b, "tensor_core")
            assert f"grid={grid_cap} " in d.plan(), d.plan()
            err = full_parity(spec, x, w, b, algo="tensor_core")
            assert err <= TOL["bf16"], f"{spec} BN={bn} KSUB={ksub} grid={grid_cap}: err={err}"


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("mode", ["im2col", "window"])
def test_full_grid_several_rounds_full_output(mode, dtype):
    """At least 3 x 152 tiles on the natural (one CTA per SM) grid, whole
    output compared: every CTA runs three or more persistent rounds."""
    spec = wl.ConvSpec("rounds_full", 96, 8, 28, 28, 64, 3, 3, 1, 1, dtype=dtype, layout="NHWC")
    x, w, b = wl.random_inputs(spec, seed=77)
    with conv2d.overrides(tc_window=1 if mode == "window" else 0, tc_cta2=0):
        y, d = run_gpu(spec, x, w, b, "tensor_core")
        assert mode in d.plan(), d.plan()
        err = full_parity(spec, x, w, b, algo="tensor_core")
    assert err <= TOL[dtype], f"{d.plan()}: err={err}"


IM2COL_SHAPES = [
    # N, C, H, W, K, R, S, stride, pad, dil, bias
    (3, 64, 9, 7, 128, 3, 3, 2, 1, 1, True),       # one M tile
    (5, 72, 13, 11, 136, 3, 3, 1, 1, 1, False),    # odd number of M tiles, ragged C and K
    (4, 128, 14, 14, 256, 3, 3, 2, 1, 1, True),    # 2 N tiles of 128
    (6, 64, 20, 20, 96, 3, 3, 1, 1, 1, True),      # K < BN
    (5, 128, 12, 12, 264, 1, 1, 1, 0, 1, True),    # 1x1 plain A, channel blocks in one box
    (3, 72, 10, 10, 64, 1, 1, 1, 0, 1, False),     # 1x1 plain A, C not a multiple of 64
    (2, 16, 17, 15, 40, 5, 5, 1, 2, 2, True),      # dilation, 5x5
]


@pytest.mark.parametrize("grid_cap", [None, 4])
@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_im2col_plain_widths_and_rounds(dtype, bn, grid_cap):
    """The im2col / plain kernel at each wide tile; with a capped grid every
    CTA runs many tiles (both accumulators, both store buffers, phase flips)."""
    with conv2d.overrides(tc_bn=bn, tc_window=0, tc_cta2=0, grid_cap=grid_cap):
        for i, (N, C, H, W, K, R, S, st, pad, dil, bias) in enumerate(IM2COL_SHAPES):
            spec = wl.ConvSpec(f"i2c{i}", N, C, H, W, K, R, S, st, pad, dil, dtype=dtype,
                               layout="NHWC", bias=bias)
            x, w, b = wl.random_inputs(spec, seed=900 + i)
            y, d = run_gpu(spec, x, w, b, "tensor_core")
            assert f"BN={bn} " in d.plan() and "window" not in d.plan(), d.plan()
            err = full_parity(spec, x, w, b, algo="tensor_core")
            assert err <= TOL[dtype], f"{spec} BN={bn} grid_cap={grid_cap}: err={err}"
    assert conv2d.get_device_status() == 0


# (BN, k-blocks per stage) of every compiled 2-CTA variant
PAIR_VARIANTS = [(128, 2), (128, 3), (128, 4), (256, 2)]


def test_pair_variant_count_matches_library():
    assert conv2d.variant_count("tensor_core_pair") == len(PAIR_VARIANTS)


@pytest.mark.parametrize("grid_cap", [None, 1, 3, 4])
@pytest.mark.parametrize("bn,ksub", PAIR_VARIANTS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_two_cta_mma(dtype, bn, ksub, grid_cap):
    """Clusters of two CTAs issuing 2-CTA MMAs (M = 256): each CTA loads its
    own A tile and half of the weight tile; with a capped grid every pair
    runs many work units, and an odd number of M tiles leaves the odd CTA's
    last tile past M."""
    with conv2d.overrides(tc_cta2=1, tc_bn=bn, tc_ksub=ksub, tc_window=0, grid_cap=grid_cap):
        for i, (N, C, H, W, K, R, S, st, pad, dil, bias) in enumerate(IM2COL_SHAPES):
            spec = wl.ConvSpec(f"c2{i}", N, C, H, W, K, R, S, st, pad, dil, dtype=dtype,
                               layout="NHWC", bias=bias)
            x, w, b = wl.random_inputs(spec, seed=950 + i)
            y, d = run_gpu(spec, x, w, b, "tensor_core")
            assert " cta2 " in d.plan() and f"BN={bn} " in d.plan() and f"ksub={ksub} " in d.plan(), d.plan()
            if grid_cap is not None:   # whole clusters of two, within the cap (at least one cluster)
                grid = int(d.plan().split("grid=")[1].split()[0])
                assert grid % 2 == 0 and 2 <= grid <= max(2, grid_cap), d.plan()
            err = full_parity(spec, x, w, b, algo="tensor_core")
            assert err <= TOL[dtype], f"{spec} BN={bn} ksub={ksub} grid_cap={grid_cap}: err={err}"
    assert conv2d.get_device_status() == 0


def test_two_cta_mma_full_grid_full_output():
    spec = wl.ConvSpec("c2_full", 96, 64, 28, 28, 128, 3, 3, 1, 1, dtype="bf16", layout="NHWC")
    x, w, b = wl.random_inputs(spec, seed=79)
    with conv2d.overrides(tc_cta2=1, tc_window=0):
        y, d = run_gpu(spec, x, w, b, "tensor_core")
        assert " cta2 " in d.plan(), d.plan()
        err = full_parity(spec, x, w, b, algo="tensor_core")
    assert err <= TOL["bf16"], f"{d.plan()}: err={err}"
    assert conv2d.get_device_status() == 0


@pytest.mark.parametrize("mode", ["single", "pair", "window"])
def test_bias_beyond_shared_staging(mode):
    """K > 2016: the epilogue reads the bias from global memory instead of its
    shared-memory copy (ragged last output-channel tile included)."""
    ovr = {"single": dict(tc_cta2=0, tc_window=0), "pair": dict(tc_cta2=1, tc_window=0),
           "window": dict(tc_window=1, tc_cta2=0)}[mode]
    with conv2d.overrides(**ovr):
        for i, (R, pad) in enumerate([(1, 0), (3, 1)]):
            spec = wl.ConvSpec(f"bigk{i}", 2, 64, 6, 7, 2072, R, R, 1, pad, 1, dtype="bf16",
                               layout="NHWC", bias=True)
            x, w, b = wl.random_inputs(spec, seed=990 + i)
            y, d = run_gpu(spec, x, w, b, "tensor_core")
            assert (" cta2 " in d.plan()) == (mode == "pair"), d.plan()
            assert ("window" in d.plan()) == (mode == "window"), d.plan()
            err = full_parity(spec, x, w, b, algo="tensor_core")
            assert err <= TOL["bf16"], f"{spec} {mode}: err={err}"
    assert conv2d.get_device_status() == 0


def test_mixed_kernels_back_to_back():
    """Four layers enqueued back to back on one stream with no host sync in
    between, on different tensor-core kernels (2-CTA clusters, window,
    single-CTA plain, 2-CTA clusters again): the programmatic dependent
    launches must hand each layer's output to the next.  Every layer is compared with the oracle on
    the input it actually received."""
    from parity import sampled_parity
    specs = [wl.ConvSpec("mix_a", 8, 128, 28, 28, 128, 7, 7, 1, 3, dtype="bf16", layout="NHWC", bias=True),
             wl.ConvSpec("mix_b", 8, 128, 28, 28, 128, 3, 3, 1, 1, dtype="bf16", layout="NHWC", bias=True),
             wl.ConvSpec("mix_c", 8, 128, 28, 28, 128, 1, 1, 1, 0, dtype="bf16", layout="NHWC", bias=True),
             wl.ConvSpec("mix_d", 8, 128, 28, 28, 128, 3, 3, 1, 1, dtype="bf16", layout="NHWC", bias=True)]
    modes = [dict(tc_cta2=1, tc_window=0), dict(tc_cta2=0, tc_window=1), dict(tc_cta2=0, tc_window=0),
             dict(tc_cta2=1, tc_window=0)]
    marks = [" cta2 ", "window", "a=tile", " cta2 "]
    x0, _, _ = wl.random_inputs(specs[0], seed=1300)
    cur = x0.cuda()
    ins, outs, params, plans = [], [], [], []
    for i, (spec, mode) in enumerate(zip(specs, modes)):
        _, w, b = wl.random_inputs(spec, seed=1301 + i)
        d = conv2d.Conv2dDesc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride,
                              spec.pad, spec.dil, spec.torch_dtype, spec.layout)
        with conv2d.overrides(**mode):
            plans.append(d.plan())
            y = d.forward(cur, w.cuda(), b.cuda())       # enqueued; no synchronisation
        ins.append(cur)
        outs.append(y)
        params.append((w, b))
        cur = y
    torch.cuda.synchronize()
    for spec, plan, mark, xin, y, (w, b) in zip(specs, plans, marks, ins, outs, params):
        assert mark in plan and (mark == " cta2 " or " cta2 " not in plan), plan
        err = sampled_parity(spec, xin.cpu(), w, b, y.cpu())
        assert err <= TOL["bf16"], f"{spec.name} ({plan}): err={err}"
    assert conv2d.get_device_status() == 0


def test_plan_reports_tensor_core():
    d = conv2d.Conv2dDesc(2, 64, 8, 8, 64, 3, 3, 1, 1, 1, torch.bfloat16, "NHWC")
    assert d.plan().startswith("tensor_core")
    assert d.workspace_bytes() == 0


def test_tensor_core_matches_cuda_core():
    spec = wl.ConvSpec("tc_vs_cc", 3, 64, 20, 20, 128, 3, 3, 1, 1, dtype="bf16", layout="NHWC")
    x, w, b = wl.random_inputs(spec, seed=5)
    y_tc, _ = run_gpu(spec, x, w, b, "tensor_core")
    y_cc, _ = run_gpu(spec, x, w, b, "cuda_core")
    diff = (y_tc.float() - y_cc.float()).abs().max().item()
    scale = y_cc.float().abs().max().item()
    assert diff <= 2 * 2 ** -8 * scale


def test_repeated_launches_are_deterministic():
    spec = wl.ConvSpec("det", 4, 128, 16, 16, 256, 3, 3, 1, 1, dtype="bf16", layout="NHWC")
    x, w, b = wl.random_inputs(spec, seed=6)
    y1, _ = run_gpu(spec, x, w, b, "tensor_core")
    y2, _ = run_gpu(spec, x, w, b, "tensor_core")
    assert torch.equal(y1, y2)
    assert conv2d.get_device_status() == 0


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("im2col", ["0", "1"])
def test_1x1_plain_and_im2col_maps(im2col, pair):
    """1x1 / stride 1 / pad 0 layers read x as a plain [N*H*W, C] matrix; the
    im2col map must give the same answer (single-CTA and 2-CTA kernels)."""
    with conv2d.overrides(tc_im2col=int(im2col), tc_cta2=pair):
        for i, (N, C, H, W, K) in enumerate([(3, 64, 7, 7, 264), (1, 72, 5, 9, 64),
                                             (4, 512, 7, 7, 256), (2, 8, 13, 11, 16)]):
            spec = wl.ConvSpec(f"p1x1_{i}", N, C, H, W, K, 1, 1, 1, 0, 1, dtype="bf16",
                               layout="NHWC", bias=bool(i % 2))
            x, w, b = wl.random_inputs(spec, seed=40 + i)
            err = full_parity(spec, x, w, b, algo="tensor_core")
            assert err <= TOL["bf16"], f"{spec}: {err}"


WINDOW_SHAPES = [
    # stride-1 layers: N, C, H, W, K, R, S, pad, dil, bias
    (1, 64, 8, 8, 64, 3, 3, 1, 1, True),
    (2, 64, 10, 12, 64, 3, 3, 1, 1, False),
    (2, 128, 9, 7, 128, 3, 3, 1, 1, True),
    (2, 64, 13, 13, 64, 5, 5, 2, 1, True),
    (1, 64, 6, 9, 64, 3, 2, 0, 2, True),           # dilation, non-square filter, no padding
    (3, 72, 11, 10, 136, 3, 3, 1, 1, True),        # channel tails, ragged K
    (2, 8, 20, 30, 24, 7, 7, 3, 1, False),         # 7x7, tiny C
    (2, 64, 5, 126, 64, 3, 3, 1, 1, True),         # padded row of 128 pixels: one row per tile
    (4, 32, 3, 3, 16, 3, 3, 1, 1, True),           # output rows fewer than rows per tile
    (2, 16, 9, 9, 32, 1, 5, 0, 1, True),           # 1 x 5 filter, no padding
]


# window-mode variants: (BN, window slot KB, resident weights), indexed as in the library
WINDOW_VARIANTS = {0: (64, 48, False), 1: (64, 48, False), 2: (128, 48, False), 3: (128, 48, False),
                   4: (256, 48, False), 5: (64, 32, False), 6: (128, 32, False), 7: (64, 32, True),
                   8: (128, 32, True), 9: (128, 25, False), 10: (128, 33, False)}


def _window_fits(shape, variant):
    N, C, H, W, K, R, S, pad, dil, bias = shape
    bn, win_kb, resident = WINDOW_VARIANTS[variant]
    wp = W + 2 * pad
    max_shift = (R - 1) * dil * wp + (S - 1) * dil
    if max_shift + 128 > win_kb * 1024 // 128:
        return False
    if resident:
        cb = (C + 63) // 64
        return K <= bn and cb * R * S * bn * 128 <= 72 * 1024
    return True


@pytest.mark.parametrize("variant", sorted(WINDOW_VARIANTS))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_window_mode(dtype, variant):
    """Stride-1 layers with one padded input window per channel block, the
    filter taps taken as row shifts of it (streamed or resident weights)."""
    ran = 0
    with conv2d.overrides(tc_window=1, tc_winvar=variant):
        for i, sh in enumerate(WINDOW_SHAPES + RESIDENT_SHAPES):
            if not _window_fits(sh, variant):
                continue
            N, C, H, W, K, R, S, pad, dil, bias = sh
            spec = wl.ConvSpec(f"win{i}", N, C, H, W, K, R, S, 1, pad, dil, dtype=dtype,
                               layout="NHWC", bias=bias)
            x, w, b = wl.random_inputs(spec, seed=200 + i)
            y, d = run_gpu(spec, x, w, b, "tensor_core")
            assert "window" in d.plan(), d.plan()
            err = full_parity(spec, x, w, b, algo="tensor_core")
            assert err <= TOL[dtype], f"{spec} variant {variant}: err={err}"
            ran += 1
    assert ran >= 3


@pytest.mark.parametrize("variant", sorted(WINDOW_VARIANTS))
def test_window_mode_many_rounds_per_cta(variant):
    """Window variants with the grid capped at 2 CTAs: many persistent rounds
    per CTA (window slots, weight stages and accumulators all wrap)."""
    ran = 0
    with conv2d.overrides(tc_window=1, tc_winvar=variant, grid_cap=2):
        for i, sh in enumerate([(5, 64, 14, 14, 64, 3, 3, 1, 1, True),
                                (4, 72, 11, 10, 120, 3, 3, 1, 1, False),
                                (6, 32, 9, 20, 40, 3, 3, 1, 1, True),
                                (4, 64, 12, 12, 128, 2, 2, 0, 1, True)]):   # fits the 128-wide resident variant
            if not _window_fits(sh, variant):
                continue
            N, C, H, W, K, R, S, pad, dil, bias = sh
            spec = wl.ConvSpec(f"winr{i}", N, C, H, W, K, R, S, 1, pad, dil, dtype="bf16",
                               layout="NHWC", bias=bias)
            x, w, b = wl.random_inputs(spec, seed=260 + i)
            y, d = run_gpu(spec, x, w, b, "tensor_core")
            assert "window" in d.plan() and "grid=2 " in d.plan(), d.plan()
            err = full_parity(spec, x, w, b, algo="tensor_core")
            assert err <= TOL["bf16"], f"{spec} variant {variant}: err={err}"
            ran += 1
    assert ran >= 1


RESIDENT_SHAPES = [
    # layers whose whole weight tensor fits one output-channel tile
    (3, 64, 14, 14, 64, 3, 3, 1, 1, True),
    (2, 32, 9, 20, 40, 3, 3, 1, 1, False),
    (2, 128, 8, 8, 64, 2, 2, 0, 1, True),
    (1, 64, 30, 40, 128, 2, 2, 1, 1, True),
    # small enough for the 128-wide resident variant (64 channels x 4 taps or fewer)
    (2, 64, 12, 12, 128, 2, 2, 0, 1, True),
    (3, 32, 10, 10, 96, 1, 3, 0, 1, False),
    (2, 64, 9, 9, 128, 2, 1, 0, 1, True),
]


def test_window_mode_not_used_where_it_cannot_apply():
    # stride 2, and a padded row longer than 128 pixels, stay on im2col
    for (H, W, st) in [(14, 14, 2), (8, 200, 1)]:
        d = conv2d.Conv2dDesc(2, 64, H, W, 64, 3, 3, st, 1, 1, torch.bfloat16, "NHWC")
        assert "a=im2col" in d.plan(), d.plan()
