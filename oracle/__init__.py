"""Oracle for the forward 2-D convolution: a plain fp64 CPU direct loop.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never loads it, and it shares no code with the CUDA
library: the arithmetic lives in ``conv2d_ref.c`` (plain C, fp64), compiled
here with gcc; this module only builds it, converts inputs exactly to fp64 in
the oracle's fixed layout, and calls it.

The definition it implements (see ``conv2d_ref.c``) follows "GPU-Accelerating
MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch Extension" (sections
"Where the Performance Bottleneck Appeared" and "Transforming Conv2D into
im2col and GEMM") and the convolution studied in "Enabling Memory-efficient
Im2win Convolution with Multi-precision Support on GPU CUDA and Tensor Cores"
(abstract):

    y[n,k,p,q] = bias[k] + sum_{c,r,s} x[n,c,p*st-pad+r*dil, q*st-pad+s*dil] * w[k,c,r,s]

Layouts accepted here: ``"NCHW"`` (x [N,C,H,W], w [K,C,R,S], y [N,K,P,Q]) and
``"NHWC"`` (x [N,H,W,C], w [K,R,S,C], y [N,P,Q,K]).  Inputs may be numpy arrays
or CPU torch tensors of any float dtype; they are widened exactly to fp64.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv2d_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build", platform.machine())
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_conv2d.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``conv2d_ref.c`` with gcc (fp64, no FMA contraction, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_out_extent.restype = _i64
    lib.oracle_out_extent.argtypes = [_i64] * 5
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_conv2d_f64.restype = ctypes.c_int
    lib.oracle_conv2d_f64.argtypes = [_dp, _dp, _dp, _dp, _dp] + [_i64] * 10 + [ctypes.c_int]
    lib.oracle_conv2d_f64_points.restype = ctypes.c_int
    lib.oracle_conv2d_f64_points.argtypes = ([_dp, _dp, _dp, ctypes.POINTER(_i64), _i64, _dp, _dp]
                                             + [_i64] * 10 + [ctypes.c_int])
    return lib


def _load(lib=None):
    """The compiled oracle, or ``lib`` when a test passes another build of it."""
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def load_build(path: str):
    """Bind another compiled copy of the oracle source (used by the mutation tests)."""
    return _bind(path)


def out_extent(size: int, ksize: int, stride: int, pad: int, dil: int, lib=None) -> int:
    """floor((size + 2*pad - dil*(ksize-1) - 1) / stride) + 1, or 0 if invalid."""
    return int(_load(lib).oracle_out_extent(size, ksize, stride, pad, dil))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _f64(a) -> np.ndarray:
    """Exact widening to a contiguous fp64 numpy array (torch or numpy input)."""
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _to_oracle_layout(x, w, bias, layout):
    x64, w64 = _f64(x), _f64(w)
    if layout == "NHWC":
        x64 = np.ascontiguousarray(x64.transpose(0, 3, 1, 2))
        w64 = np.ascontiguousarray(w64.transpose(0, 3, 1, 2))
    elif layout != "NCHW":
        raise ValueError(f"layout must be NCHW or NHWC, got {layout!r}")
    if x64.ndim != 4 or w64.ndim != 4 or x64.shape[1] != w64.shape[1]:
        raise ValueError(f"bad shapes x{x64.shape} w{w64.shape}")
    b64 = None if bias is None else _f64(bias).reshape(-1)
    if b64 is not None and b64.shape[0] != w64.shape[0]:
        raise ValueError("bias must have K entries")
    return x64, w64, b64


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def conv2d(x, w, bias=None, stride=1, pad=0, dil=1, layout="NCHW", threads=0, lib=None):
    """Full output (y, den) in fp64, laid out like ``layout``."""
    x64, w64, b64 = _to_oracle_layout(x, w, bias, layout)
    N, C, H, W = x64.shape
    K, _, R, S = w64.shape
    P, Q = out_extent(H, R, stride, pad, dil, lib), out_extent(W, S, stride, pad, dil, lib)
    if P < 1 or Q < 1:
        raise ValueError("empty output")
    y = np.empty((N, K, P, Q), dtype=np.float64)
    den = np.empty_like(y)
    rc = _load(lib).oracle_conv2d_f64(_ptr(x64), _ptr(w64), _ptr(b64), _ptr(y), _ptr(den),
                                   N, C, H, W, K, R, S, stride, pad, dil, int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the shape (rc={rc})")
    if layout == "NHWC":
        y, den = y.transpose(0, 2, 3, 1), den.transpose(0, 2, 3, 1)
    return np.ascontiguousarray(y), np.ascontiguousarray(den)


def conv2d_points(x, w, bias, idx, stride=1, pad=0, dil=1, layout="NCHW", threads=0, lib=None):
    """Outputs at logical indices idx[i] = (n, k, p, q): returns (y, den) of shape [len(idx)]."""
    x64, w64, b64 = _to_oracle_layout(x, w, bias, layout)
    N, C, H, W = x64.shape
    K, _, R, S = w64.shape
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64).reshape(-1, 4))
    y = np.empty(idx.shape[0], dtype=np.float64)
    den = np.empty_like(y)
    rc = _load(lib).oracle_conv2d_f64_points(_ptr(x64), _ptr(w64), _ptr(b64),
                                          idx.ctypes.data_as(ctypes.POINTER(_i64)), idx.shape[0],
                                          _ptr(y), _ptr(den), N, C, H, W, K, R, S,
                                          stride, pad, dil, int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the request (rc={rc})")
    return y, den


def error_ratio(y_test, y_ref, den) -> float:
    """max |y_test - y_ref| / den over all outputs (fp64).

    Where den == 0 (every tap in padding and no bias) the exact answer is 0 and
    any nonzero y_test counts as an infinite error.
    """
    yt = _f64(y_test)
    diff = np.abs(yt - np.asarray(y_ref, dtype=np.float64))
    den = np.asarray(den, dtype=np.float64)
    if not np.all(np.isfinite(yt)):
        return float("inf")
    zero = den == 0
    if np.any(diff[zero] != 0):
        return float("inf")
    if diff.size == 0:
        return 0.0
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(zero, 0.0, diff / np.where(zero, 1.0, den))
    return float(ratio.max())
