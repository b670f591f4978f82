"""Host-only checks of the C ABI: the library loads, exports what the header
declares, and validates arguments before any launch.  No kernel runs here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "conv2d.h")


@pytest.fixture(scope="module")
def lib():
    from cnn_convolution_gb300 import build, conv2d
    build.build()
    return conv2d.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(conv2d_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("conv2d_desc_create", "conv2d_workspace_bytes", "conv2d_forward",
                     "conv2d_desc_destroy", "conv2d_output_dims", "conv2d_get_device_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in conv2d.h but not exported"


def test_nm_shows_c_linkage():
    from cnn_convolution_gb300 import build
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (conv2d_\w+)", out))
    assert set(declared_functions()) <= exported


def _desc(lib, *args):
    h = ctypes.c_void_p()
    rc = lib.conv2d_desc_create(ctypes.byref(h), *args)
    return rc, h


def test_desc_output_dims_and_workspace(lib, oracle_mod):
    cases = [(256, 3, 30, 30, 32, 3, 3, 1, 1, 1), (256, 32, 30, 30, 64, 3, 3, 2, 1, 1),
             (256, 64, 15, 15, 128, 2, 2, 2, 1, 1), (256, 128, 8, 8, 256, 2, 2, 2, 0, 1),
             (128, 64, 56, 56, 64, 3, 3, 1, 1, 1), (64, 128, 28, 28, 128, 7, 7, 1, 3, 1),
             (256, 256, 14, 14, 512, 3, 3, 2, 1, 1), (2, 5, 9, 13, 7, 3, 2, 3, 2, 2)]
    for c in cases:
        for dtype in (0, 1, 2):
            for layout in (0, 1):
                rc, h = _desc(lib, *c, dtype, layout)
                assert rc == 0
                P, Q = ctypes.c_int(), ctypes.c_int()
                assert lib.conv2d_output_dims(h, ctypes.byref(P), ctypes.byref(Q)) == 0
                N, C, H, W, K, R, S, st, pad, dil = c
                assert P.value == oracle_mod.out_extent(H, R, st, pad, dil)
                assert Q.value == oracle_mod.out_extent(W, S, st, pad, dil)
                ws = ctypes.c_size_t(123)
                assert lib.conv2d_workspace_bytes(h, ctypes.byref(ws)) == 0
                assert ws.value == 0
                assert lib.conv2d_desc_destroy(h) == 0


BAD_SHAPES = [
    (0, 3, 30, 30, 32, 3, 3, 1, 1, 1),     # N = 0
    (1, 0, 30, 30, 32, 3, 3, 1, 1, 1),     # C = 0
    (1, 3, 0, 30, 32, 3, 3, 1, 1, 1),      # H = 0
    (1, 3, 30, 30, 0, 3, 3, 1, 1, 1),      # K = 0
    (1, 3, 30, 30, 32, 0, 3, 1, 1, 1),     # R = 0
    (1, 3, 30, 30, 32, 3, 3, 0, 1, 1),     # stride = 0
    (1, 3, 30, 30, 32, 3, 3, 1, -1, 1),    # pad < 0
    (1, 3, 30, 30, 32, 3, 3, 1, 1, 0),     # dil = 0
    (1, 3, 2, 2, 32, 5, 5, 1, 0, 1),       # filter larger than the padded input: P <= 0
    (1, 3, 5, 5, 32, 3, 3, 1, 0, 3),       # dilated filter too wide
    (1 << 20, 1 << 10, 1 << 10, 1 << 10, 1, 1, 1, 1, 0, 1),   # element count overflow
]


@pytest.mark.parametrize("shape", BAD_SHAPES)
def test_invalid_shapes_rejected(lib, shape):
    rc, h = _desc(lib, *shape, 0, 0)
    assert rc == 1 and not h.value


def test_invalid_dtype_layout_rejected(lib):
    assert _desc(lib, 1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 7, 0)[0] == 1
    assert _desc(lib, 1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 0, 5)[0] == 1


def test_null_arguments(lib):
    assert lib.conv2d_desc_create(None, 1, 1, 1, 1, 1, 1, 1, 1, 0, 1, 0, 0) == 1
    assert lib.conv2d_output_dims(None, None, None) == 1
    assert lib.conv2d_workspace_bytes(None, None) == 1
    assert lib.conv2d_desc_destroy(None) == 0
    # null tensors are rejected before any CUDA call is needed
    assert lib.conv2d_forward(None, None, None, None, 1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 0, 0, None) == 1


def test_forward_rejects_bad_shape_before_launch(lib):
    # P <= 0: rejected in validation even with non-null (never dereferenced) pointers
    rc = lib.conv2d_forward(ctypes.c_void_p(16), ctypes.c_void_p(32), None, ctypes.c_void_p(64),
                            1, 3, 2, 2, 4, 5, 5, 1, 0, 1, 0, 0, None)
    assert rc == 1


def test_misaligned_pointer_rejected_before_launch(lib):
    # fp32 tensors at odd addresses fail the alignment check, which precedes any CUDA call
    rc = lib.conv2d_forward(ctypes.c_void_p(0x1001), ctypes.c_void_p(0x2000), None,
                            ctypes.c_void_p(0x100000), 1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 0, 0, None)
    assert rc == 3


def test_aliasing_rejected_before_launch(lib):
    # y overlapping x (same base) is an argument error, found before any CUDA call
    rc = lib.conv2d_forward(ctypes.c_void_p(0x10000), ctypes.c_void_p(0x90000), None,
                            ctypes.c_void_p(0x10000), 1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 0, 0, None)
    assert rc == 1


def test_status_strings(lib):
    for code in range(7):
        assert lib.conv2d_status_string(code)
    assert lib.conv2d_status_string(99) == b"unknown status"


def test_set_algo_validation(lib):
    rc, h = _desc(lib, 2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 0, 0)
    assert rc == 0
    assert lib.conv2d_desc_set_algo(h, 1) == 0
    assert lib.conv2d_desc_set_algo(h, 9) == 1
    # fp32 (either layout) has the split-precision tensor-core kernel
    assert lib.conv2d_desc_set_algo(h, 2) == 0
    lib.conv2d_desc_destroy(h)
    # fp16 NCHW has no tensor-core kernel
    rc, h = _desc(lib, 2, 8, 8, 8, 8, 3, 3, 1, 1, 1, 1, 0)
    assert rc == 0
    assert lib.conv2d_desc_set_algo(h, 2) == 2
    lib.conv2d_desc_destroy(h)


def test_python_binding_fails_loudly_without_library(tmp_path):
    from cnn_convolution_gb300 import conv2d
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        conv2d.load(str(tmp_path / "missing.so"))
    conv2d._lib = None   # reload the real library for later tests


def test_overrides_set_get_and_validation(lib):
    from cnn_convolution_gb300 import conv2d
    assert conv2d.get_override("tc_bn") is None
    with conv2d.overrides(tc_bn=128, grid_cap=3):
        assert conv2d.get_override("tc_bn") == 128
        assert conv2d.get_override("grid_cap") == 3
    assert conv2d.get_override("tc_bn") is None
    assert conv2d.get_override("grid_cap") is None
    v = ctypes.c_int()
    assert lib.conv2d_set_override(99, 1) == 1            # unknown key
    assert lib.conv2d_set_override(-1, 1) == 1
    assert lib.conv2d_set_override(0, -2) == 1            # below -1
    assert lib.conv2d_get_override(99, ctypes.byref(v)) == 1
    assert lib.conv2d_get_override(0, None) == 1
    assert len(conv2d.OVERRIDES) == 16                    # CONV2D_OVR_COUNT in the header
    text = open(HEADER).read()
    body = text[text.index("typedef enum {\n    CONV2D_OVR_DIRECT"):text.index("CONV2D_OVR_COUNT")]
    names = re.findall(r"CONV2D_OVR_([A-Z0-9_]+)", body)
    assert [n.lower() for n in names] == list(conv2d.OVERRIDES)


def test_overrides_are_seeded_from_the_environment_once():
    """The environment is read at the first use only; later changes of it have no effect."""
    import subprocess
    import sys
    code = ("import os, sys; sys.path.insert(0, %r)\n"
            "from cnn_convolution_gb300 import conv2d\n"
            "a = conv2d.get_override('tc_bn')\n"
            "os.environ['CONV2D_TC_BN'] = '64'\n"
            "b = conv2d.get_override('tc_bn')\n"
            "print(a, b, conv2d.get_override('tf_var'))\n") % ROOT
    env = dict(os.environ, CONV2D_TC_BN="256")
    env.pop("CONV2D_TF_VAR", None)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True).stdout.split()
    assert out == ["256", "256", "None"]


def test_variant_counts(lib):
    from cnn_convolution_gb300 import conv2d
    counts = {f: conv2d.variant_count(f) for f in conv2d.FAMILIES}
    import parity
    assert counts == {"cuda_core_tile": 8, "tensor_core": 7, "tensor_core_window": 11,
                      "tf32x3": parity.N_TF_VARIANTS, "tensor_core_pair": 4}
    n = ctypes.c_int()
    assert lib.conv2d_variant_count(7, ctypes.byref(n)) == 1
    assert lib.conv2d_variant_count(0, None) == 1
