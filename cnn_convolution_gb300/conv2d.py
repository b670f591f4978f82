"""Thin Python binding of libconv2d_gb300 (argument marshalling only).

Every step of the convolution runs in the library's CUDA kernels; this
module only checks that torch tensors are dense CUDA tensors of one dtype,
passes their device pointers and the current CUDA stream through the C ABI
declared in include/conv2d.h, and turns status codes into exceptions.  There
is no fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from contextlib import contextmanager
from typing import Optional, Tuple

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2
NCHW, NHWC = 0, 1
ALGO_AUTO, ALGO_CUDA_CORE, ALGO_TENSOR_CORE = 0, 1, 2

_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
_LAYOUT_CODE = {"NCHW": NCHW, "NHWC": NHWC}
_ALGO_CODE = {"auto": ALGO_AUTO, "cuda_core": ALGO_CUDA_CORE, "tensor_core": ALGO_TENSOR_CORE}

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "misaligned pointer",
          4: "CUDA error", 5: "kernel barrier wait timed out", 6: "internal error"}


class Conv2dError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, 'unknown')} (status {code})")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None):
    """Load the compiled library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or _build.LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build it with cnn_convolution_gb300.build.build() "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(p)
            _declare(lib)
            _lib = lib
    return _lib


def _declare(lib):
    c_int, vp, i32 = ctypes.c_int, ctypes.c_void_p, ctypes.c_int
    lib.conv2d_desc_create.restype = c_int
    lib.conv2d_desc_create.argtypes = [ctypes.POINTER(vp)] + [i32] * 10 + [c_int, c_int]
    lib.conv2d_desc_destroy.restype = c_int
    lib.conv2d_desc_destroy.argtypes = [vp]
    lib.conv2d_output_dims.restype = c_int
    lib.conv2d_output_dims.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.conv2d_workspace_bytes.restype = c_int
    lib.conv2d_workspace_bytes.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
    lib.conv2d_desc_set_algo.restype = c_int
    lib.conv2d_desc_set_algo.argtypes = [vp, c_int]
    lib.conv2d_desc_plan.restype = c_int
    lib.conv2d_desc_plan.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
    lib.conv2d_forward_desc.restype = c_int
    lib.conv2d_forward_desc.argtypes = [vp, vp, vp, vp, vp, vp]
    lib.conv2d_forward.restype = c_int
    lib.conv2d_forward.argtypes = [vp, vp, vp, vp] + [i32] * 10 + [c_int, c_int, vp]
    lib.conv2d_status_string.restype = ctypes.c_char_p
    lib.conv2d_status_string.argtypes = [c_int]
    lib.conv2d_get_device_status.restype = c_int
    lib.conv2d_get_device_status.argtypes = []
    lib.conv2d_version.restype = c_int
    lib.conv2d_version.argtypes = []
    lib.conv2d_deconv_output_dims.restype = c_int
    lib.conv2d_deconv_output_dims.argtypes = [i32] * 8 + [ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.conv2d_deconv_forward.restype = c_int
    lib.conv2d_deconv_forward.argtypes = [vp] * 4 + [i32] * 11 + [c_int, c_int, vp]
    lib.conv2d_convlstm_cell.restype = c_int
    lib.conv2d_convlstm_cell.argtypes = [vp] * 6 + [i32] * 9 + [ctypes.c_longlong, vp]
    lib.conv2d_set_override.restype = c_int
    lib.conv2d_set_override.argtypes = [c_int, c_int]
    lib.conv2d_get_override.restype = c_int
    lib.conv2d_get_override.argtypes = [c_int, ctypes.POINTER(c_int)]
    lib.conv2d_variant_count.restype = c_int
    lib.conv2d_variant_count.argtypes = [c_int, ctypes.POINTER(c_int)]
    lib.conv2d_peak_probe.restype = c_int
    lib.conv2d_peak_probe.argtypes = [c_int, c_int, vp, ctypes.POINTER(ctypes.c_double)]
    lib.conv2d_signature_matrices.restype = c_int
    lib.conv2d_signature_matrices.argtypes = [vp, i32, i32, ctypes.POINTER(i32), i32, i32, i32,
                                              vp, vp]


def _check(code: int, what: str):
    if code != 0:
        raise Conv2dError(code, what)


class Conv2dDesc:
    """A layer descriptor (sizes, dtype, layout) owned by this object."""

    def __init__(self, N, C, H, W, K, R, S, stride=1, pad=0, dil=1,
                 dtype: torch.dtype = torch.float32, layout: str = "NCHW"):
        self._lib = load()
        self.sizes = (N, C, H, W, K, R, S, stride, pad, dil)
        self.dtype, self.layout = dtype, layout
        h = ctypes.c_void_p()
        _check(self._lib.conv2d_desc_create(ctypes.byref(h), N, C, H, W, K, R, S, stride, pad, dil,
                                            _DTYPE_CODE[dtype], _LAYOUT_CODE[layout]),
               "conv2d_desc_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.conv2d_desc_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def output_dims(self) -> Tuple[int, int]:
        P, Q = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.conv2d_output_dims(self._h, ctypes.byref(P), ctypes.byref(Q)),
               "conv2d_output_dims")
        return P.value, Q.value

    def workspace_bytes(self) -> int:
        b = ctypes.c_size_t()
        _check(self._lib.conv2d_workspace_bytes(self._h, ctypes.byref(b)), "conv2d_workspace_bytes")
        return b.value

    def set_algo(self, algo: str):
        _check(self._lib.conv2d_desc_set_algo(self._h, _ALGO_CODE[algo]), "conv2d_desc_set_algo")

    def plan(self) -> str:
        buf = ctypes.create_string_buffer(256)
        _check(self._lib.conv2d_desc_plan(self._h, buf, 256), "conv2d_desc_plan")
        return buf.value.decode()

    def y_shape(self):
        shape = getattr(self, "_y_shape", None)
        if shape is None:
            N, C, H, W, K = self.sizes[:5]
            P, Q = self.output_dims()
            shape = (N, K, P, Q) if self.layout == "NCHW" else (N, P, Q, K)
            self._y_shape = shape
        return shape

    def forward(self, x, w, bias=None, y=None, stream=None):
        if y is None:
            y = torch.empty(self.y_shape(), dtype=self.dtype, device=x.device)
        dt = self.dtype
        # dtype and density are the caller's promise the library cannot see;
        # device placement it checks itself (host pointers are rejected)
        if not (x.dtype is dt and w.dtype is dt and y.dtype is dt and (bias is None or bias.dtype is dt)):
            _validate(x, w, bias, y, dt)        # raises with the exact reason
        if not (x.is_contiguous() and w.is_contiguous() and y.is_contiguous()
                and (bias is None or bias.is_contiguous())):
            _validate(x, w, bias, y, dt)
        code = self._lib.conv2d_forward_desc(self._h, x.data_ptr(), w.data_ptr(),
                                             None if bias is None else bias.data_ptr(),
                                             y.data_ptr(), _stream_handle(stream, x.device))
        if code:
            _validate(x, w, bias, y, dt)
            _check(code, "conv2d_forward_desc")
        return y


def _validate(x, w, bias, y, dtype):
    for name, t in (("x", x), ("w", w), ("y", y)) + ((("bias", bias),) if bias is not None else ()):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != dtype:
            raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, device):
    """The cudaStream_t to launch on: `stream`'s, or the current stream of
    `device` (read through torch's raw-stream query, which costs a fraction
    of building a Stream object)."""
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:
        idx = device.index if device.index is not None else torch.cuda.current_device()
        return ctypes.c_void_p(_raw_stream(idx))
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def output_dims(H, W, R, S, stride=1, pad=0, dil=1) -> Tuple[int, int]:
    d = Conv2dDesc(1, 1, H, W, 1, R, S, stride, pad, dil)
    return d.output_dims()


def forward(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None,
            stride: int = 1, pad: int = 0, dil: int = 1, layout: str = "NCHW",
            y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = conv2d(x, w) + bias through conv2d_forward (plan chosen per shape).

    layout "NCHW": x [N,C,H,W], w [K,C,R,S] -> y [N,K,P,Q];
    layout "NHWC": x [N,H,W,C], w [K,R,S,C] -> y [N,P,Q,K].
    """
    lib = load()
    if layout == "NCHW":
        N, C, H, W = x.shape
        K, C2, R, S = w.shape
    elif layout == "NHWC":
        N, H, W, C = x.shape
        K, R, S, C2 = w.shape
    else:
        raise ValueError(layout)
    if C2 != C:
        raise ValueError("x and w disagree on C")
    if y is None:
        d = Conv2dDesc(N, C, H, W, K, R, S, stride, pad, dil, x.dtype, layout)
        y = torch.empty(d.y_shape(), dtype=x.dtype, device=x.device)
    _validate(x, w, bias, y, x.dtype)
    st = _stream_handle(stream, x.device)
    _check(lib.conv2d_forward(x.data_ptr(), w.data_ptr(),
                              None if bias is None else bias.data_ptr(), y.data_ptr(),
                              N, C, H, W, K, R, S, stride, pad, dil,
                              _DTYPE_CODE[x.dtype], _LAYOUT_CODE[layout], st), "conv2d_forward")
    return y


def signature_matrices(series: torch.Tensor, windows, t_first: int, n_steps: int,
                       out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """MSCRED signature matrices through conv2d_signature_matrices.

    series: CUDA fp32 [n_signals, T]; returns fp32 [n_steps, len(windows),
    n_signals, n_signals] with out[b, c] = the Gram matrix of the last
    windows[c] samples before time t_first + b, divided by windows[c] (the
    NCHW input of the encoder's first convolution).
    """
    lib = load()
    if not isinstance(series, torch.Tensor) or not series.is_cuda or series.dtype != torch.float32:
        raise ValueError("series must be a CUDA float32 tensor")
    if series.dim() != 2 or not series.is_contiguous():
        raise ValueError("series must be a contiguous [n_signals, T] tensor")
    n, T = series.shape
    wins = [int(w) for w in windows]
    shape = (n_steps, len(wins), n, n)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=series.device)
    elif tuple(out.shape) != shape or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous float32 tensor of shape {shape}")
    warr = (ctypes.c_int * max(1, len(wins)))(*wins)
    _check(lib.conv2d_signature_matrices(series.data_ptr(), n, T, warr, len(wins), t_first, n_steps,
                                         out.data_ptr(), _stream_handle(stream, series.device)),
           "conv2d_signature_matrices")
    return out


def convlstm_cell(xh: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                  c_prev: torch.Tensor, pad: int, dil: int = 1,
                  c_next: Optional[torch.Tensor] = None, h_next: Optional[torch.Tensor] = None,
                  h_img_stride: Optional[int] = None, stream=None):
    """One ConvLSTM cell step through conv2d_convlstm_cell (fp32, NCHW).

    xh [N, Cx+Ch, H, W] = [x_t, h_{t-1}]; w [4Ch, Cx+Ch, R, S] with gates
    (i, f, o, g); c_prev [N, Ch, H, W].  Returns (c_next, h_next).  h_next may
    be a view into another buffer: pass its first element's tensor and
    h_img_stride, the element distance between its images.
    """
    lib = load()
    N, C, H, W = xh.shape
    K, C2, R, S = w.shape
    Ch = K // 4
    if C2 != C or K % 4 or tuple(c_prev.shape) != (N, Ch, H, W):
        raise ValueError("shapes of xh, w and c_prev disagree")
    for name, t in (("xh", xh), ("w", w), ("c_prev", c_prev)) + ((("bias", bias),) if bias is not None else ()):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor")
    if c_next is None:
        c_next = torch.empty_like(c_prev)
    if h_next is None:
        h_next = torch.empty_like(c_prev)
    if h_img_stride is None:
        h_img_stride = Ch * H * W
    _check(lib.conv2d_convlstm_cell(xh.data_ptr(), w.data_ptr(),
                                    None if bias is None else bias.data_ptr(), c_prev.data_ptr(),
                                    c_next.data_ptr(), h_next.data_ptr(), N, C - Ch, Ch, H, W, R, S,
                                    pad, dil, int(h_img_stride), _stream_handle(stream, xh.device)),
           "conv2d_convlstm_cell")
    return c_next, h_next


def deconv_output_dims(P, Q, R, S, stride=1, pad=0, dil=1, out_pad=0) -> Tuple[int, int]:
    lib = load()
    H, W = ctypes.c_int(), ctypes.c_int()
    _check(lib.conv2d_deconv_output_dims(P, Q, R, S, stride, pad, dil, out_pad,
                                         ctypes.byref(H), ctypes.byref(W)), "conv2d_deconv_output_dims")
    return H.value, W.value


def deconv_forward(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None,
                   stride: int = 1, pad: int = 0, dil: int = 1, out_pad: int = 0,
                   y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Transposed convolution through conv2d_deconv_forward (fp32 NCHW).

    x [N, K, P, Q], w [K, C, R, S] -> y [N, C, H, W]."""
    lib = load()
    N, K, P, Q = x.shape
    K2, C, R, S = w.shape
    if K2 != K:
        raise ValueError("x and w disagree on K")
    H, W = deconv_output_dims(P, Q, R, S, stride, pad, dil, out_pad)
    if y is None:
        y = torch.empty((N, C, H, W), dtype=x.dtype, device=x.device)
    _validate(x, w, bias, y, x.dtype)
    _check(lib.conv2d_deconv_forward(x.data_ptr(), w.data_ptr(),
                                     None if bias is None else bias.data_ptr(), y.data_ptr(),
                                     N, K, P, Q, C, R, S, stride, pad, dil, out_pad,
                                     _DTYPE_CODE[x.dtype], _LAYOUT_CODE["NCHW"],
                                     _stream_handle(stream, x.device)), "conv2d_deconv_forward")
    return y


# Process-wide chooser overrides (conv2d_set_override), by the names of their
# enum constants without the CONV2D_OVR_ prefix, lower case.
OVERRIDES = {name: i for i, name in enumerate(
    ["direct", "cc_tile", "cc_split", "tc_bn", "tc_ksub", "tc_im2col", "tc_window", "tc_winvar",
     "tc_rotate", "tf_var", "fp32_tc", "deconv_tc", "grid_cap", "test_withhold",
     "test_wait_kcycles", "tc_cta2"])}
FAMILIES = {"cuda_core_tile": 0, "tensor_core": 1, "tensor_core_window": 2, "tf32x3": 3,
            "tensor_core_pair": 4}


def set_override(name: str, value: Optional[int]):
    """Set (or, with None, clear) one chooser override for the whole process."""
    _check(load().conv2d_set_override(OVERRIDES[name], -1 if value is None else int(value)),
           f"conv2d_set_override({name})")


def get_override(name: str) -> Optional[int]:
    v = ctypes.c_int()
    _check(load().conv2d_get_override(OVERRIDES[name], ctypes.byref(v)), "conv2d_get_override")
    return None if v.value == -1 else v.value


@contextmanager
def overrides(**kw):
    """Set overrides for the duration of a with-block, then restore the old values."""
    old = {k: get_override(k) for k in kw}
    try:
        for k, v in kw.items():
            set_override(k, v)
        yield
    finally:
        for k, v in old.items():
            set_override(k, v)


def variant_count(family: str) -> int:
    """Number of compiled variants of a kernel family."""
    n = ctypes.c_int()
    _check(load().conv2d_variant_count(FAMILIES[family], ctypes.byref(n)), "conv2d_variant_count")
    return n.value


PEAK_KINDS = {"ffma": 0, "tf32_mma": 1, "bf16_mma": 2}


def peak_probe(kind: str, iters: int, stream=None) -> float:
    """Launch one throughput-probe kernel on the current stream; returns its FLOPs."""
    f = ctypes.c_double()
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(load().conv2d_peak_probe(PEAK_KINDS[kind], int(iters), _stream_handle(stream, dev),
                                    ctypes.byref(f)), f"conv2d_peak_probe({kind})")
    return f.value


def get_device_status() -> int:
    return load().conv2d_get_device_status()


def version() -> int:
    return load().conv2d_version()
