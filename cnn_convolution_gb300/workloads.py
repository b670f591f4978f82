"""Seeded synthetic workloads: shapes and input generators.

This module holds no convolution arithmetic.  It only names the layer shapes
that are measured and tested and draws their inputs (x, w, bias) from seeded
generators, so that the CUDA path and the oracle see the same values.

Values are always drawn in logical NCHW / KCRS order and in fp32 (fp64 for
the signature matrices), then rounded once to the layer's dtype on the CPU and
finally permuted to NHWC / KRSC when the layer is channels-last.  A given seed
therefore gives the same logical values in either layout.

Seeds: 1000*workload + {0: x, 1: w, 2: bias} + 10*sub-index (the encoder's
layer, or the kernel-size / layer variant).

The MSCRED inputs follow "GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and
a Custom PyTorch Extension" ("Why Signature Matrices Are Useful": pairwise
products of signals over windows of several lengths; "Experimental Setup":
30 features).  The industrial data set of that page is confidential, so
seeded random-walk signals stand in for it.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class ConvSpec:
    """One convolution layer: sizes, hyper-parameters, dtype and layout."""
    name: str
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    stride: int = 1
    pad: int = 0
    dil: int = 1
    dtype: str = "f32"          # "f32" | "f16" | "bf16"
    layout: str = "NCHW"        # "NCHW" | "NHWC"
    bias: bool = True

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def x_shape(self) -> Tuple[int, ...]:
        if self.layout == "NCHW":
            return (self.N, self.C, self.H, self.W)
        return (self.N, self.H, self.W, self.C)

    def w_shape(self) -> Tuple[int, ...]:
        if self.layout == "NCHW":
            return (self.K, self.C, self.R, self.S)
        return (self.K, self.R, self.S, self.C)

    def replace(self, **kw) -> "ConvSpec":
        return dataclasses.replace(self, **kw)


# --------------------------------------------------------------------------
# element distributions (logical NCHW / KCRS order, fp32)
# --------------------------------------------------------------------------

def _uniform(seed: int, shape, lo: float, hi: float) -> np.ndarray:
    return np.random.default_rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def _normal(seed: int, shape, std: float) -> np.ndarray:
    return (np.random.default_rng(seed).standard_normal(size=shape) * std).astype(np.float32)


def _finish(a: np.ndarray, spec: ConvSpec, kind: str) -> torch.Tensor:
    """Round once to the layer dtype, then permute to the layer's layout."""
    t = torch.from_numpy(np.ascontiguousarray(a)).to(spec.torch_dtype)
    if spec.layout == "NHWC" and kind in ("x", "w"):
        t = t.permute(0, 2, 3, 1)
    return t.contiguous()


def random_walk_series(n_signals: int, length: int, seed: int) -> np.ndarray:
    """Seeded random walks s_i(t) = cumulative sum of N(0,1) steps, fp64 [n_signals, length]."""
    rng = np.random.default_rng(seed)
    return np.cumsum(rng.standard_normal(size=(n_signals, length)), axis=1)


def mscred_encoder_series(n: int = 256) -> torch.Tensor:
    """The raw signals behind ``mscred_encoder_input(n)``: fp32 [30, 60 + n - 1]."""
    return torch.from_numpy(random_walk_series(MSCRED_SIGNALS, 60 + n - 1, 1000).astype(np.float32))


def signature_matrices(n_signals: int, length: int, windows: Tuple[int, ...],
                       end_times: List[int], seed: int) -> np.ndarray:
    """MSCRED-style signature matrices, fp64, shape [len(end_times), len(windows), n, n].

    Signals are seeded random walks s_i(t) = cumulative sum of N(0,1) steps,
    t = 0..length-1.  For an end time e and window w the matrix is
    M_ij = sum_{t=e-w}^{e-1} s_i(t) s_j(t) / w.
    """
    sig = random_walk_series(n_signals, length, seed)
    out = np.empty((len(end_times), len(windows), n_signals, n_signals), dtype=np.float64)
    for b, e in enumerate(end_times):
        for c, win in enumerate(windows):
            seg = sig[:, e - win:e]
            out[b, c] = (seg @ seg.T) / win
    return out


# --------------------------------------------------------------------------
# the measured workloads
# --------------------------------------------------------------------------

MSCRED_WINDOWS = (10, 30, 60)
MSCRED_SIGNALS = 30

MSCRED_SINGLE = ConvSpec("mscred_sig_conv_n1_c3_30x30_k32_3x3", N=1, C=3, H=30, W=30, K=32,
                         R=3, S=3, stride=1, pad=1, dtype="f32", layout="NCHW", bias=True)

MSCRED_ENCODER = [
    ConvSpec("mscred_enc_l1_n256_c3_30x30_k32_3x3s1p1", 256, 3, 30, 30, 32, 3, 3, 1, 1),
    ConvSpec("mscred_enc_l2_n256_c32_30x30_k64_3x3s2p1", 256, 32, 30, 30, 64, 3, 3, 2, 1),
    ConvSpec("mscred_enc_l3_n256_c64_15x15_k128_2x2s2p1", 256, 64, 15, 15, 128, 2, 2, 2, 1),
    ConvSpec("mscred_enc_l4_n256_c128_8x8_k256_2x2s2p0", 256, 128, 8, 8, 256, 2, 2, 2, 0),
]

CNN_MID_F16 = ConvSpec("cnn_mid_f16_nhwc_n128_c64_56x56_k64_3x3", 128, 64, 56, 56, 64, 3, 3,
                       1, 1, dtype="f16", layout="NHWC", bias=True)

KSWEEP_BF16 = [ConvSpec(f"ksweep_bf16_nhwc_n64_c128_28x28_k128_{r}x{r}", 64, 128, 28, 28, 128,
                        r, r, 1, (r - 1) // 2, dtype="bf16", layout="NHWC", bias=False)
               for r in (1, 3, 5, 7)]

DEEP_BF16 = [
    ConvSpec("deep_bf16_nhwc_n256_c256_14x14_k512_3x3s2p1", 256, 256, 14, 14, 512, 3, 3, 2, 1,
             dtype="bf16", layout="NHWC", bias=False),
    ConvSpec("deep_bf16_nhwc_n256_c512_7x7_k2048_1x1", 256, 512, 7, 7, 2048, 1, 1, 1, 0,
             dtype="bf16", layout="NHWC", bias=False),
]


def mscred_single_inputs(spec: ConvSpec = MSCRED_SINGLE):
    """Single signature-matrix conv: series of 60 steps, the final time step."""
    seed = 0
    x = signature_matrices(MSCRED_SIGNALS, 60, MSCRED_WINDOWS, [60], seed)
    b = 1.0 / math.sqrt(spec.C * spec.R * spec.S)
    w = _uniform(seed + 1, (spec.K, spec.C, spec.R, spec.S), -b, b)
    bias = _uniform(seed + 2, (spec.K,), -b, b)
    return (_finish(x.astype(np.float32), spec, "x"), _finish(w, spec, "w"),
            _finish(bias, spec, "b"))


def mscred_encoder_input(n: int = 256) -> torch.Tensor:
    """n time steps of 3x30x30 signature matrices (end times 60 .. 60+n-1)."""
    seed = 1000
    x = signature_matrices(MSCRED_SIGNALS, 60 + n - 1, MSCRED_WINDOWS,
                           list(range(60, 60 + n)), seed)
    return _finish(x.astype(np.float32), MSCRED_ENCODER[0].replace(N=n), "x")


def kaiming_params(spec: ConvSpec, seed: int):
    """Kaiming-uniform: w ~ U(+-sqrt(6/fan_in)), bias ~ U(+-1/sqrt(fan_in))."""
    fan_in = spec.C * spec.R * spec.S
    wb = math.sqrt(6.0 / fan_in)
    bb = 1.0 / math.sqrt(fan_in)
    w = _uniform(seed + 1, (spec.K, spec.C, spec.R, spec.S), -wb, wb)
    bias = _uniform(seed + 2, (spec.K,), -bb, bb)
    return _finish(w, spec, "w"), _finish(bias, spec, "b")


def mscred_encoder_params():
    """Weights and biases of the 4 encoder layers (seeds 1000 + 10*layer)."""
    return [kaiming_params(spec, 1000 + 10 * i) for i, spec in enumerate(MSCRED_ENCODER)]


def layer_inputs(spec: ConvSpec, workload: int, sub: int = 0, dist: Optional[str] = None):
    """x, w, bias (bias None when spec.bias is False) for a tensor-core workload.

    dist selects the distribution family: "mid" (U(-1,1)/sqrt(CRS) for x and
    w, U(-0.1,0.1) bias), "normal" (x ~ N(0,1), w ~ N(0, 1/CRS)), "relu"
    (x = max(N(0,1), 0), w ~ N(0, 2/CRS)), "positive" (x, w ~ U(0,1): every
    product has the same sign, the hardest case for the error ratio).
    """
    seed = 1000 * workload + 10 * sub
    crs = spec.C * spec.R * spec.S
    xs = (spec.N, spec.C, spec.H, spec.W)
    ws = (spec.K, spec.C, spec.R, spec.S)
    dist = dist or "normal"
    if dist == "mid":
        x = _uniform(seed, xs, -1.0, 1.0) / np.float32(math.sqrt(crs))
        w = _uniform(seed + 1, ws, -1.0, 1.0) / np.float32(math.sqrt(crs))
        bias = _uniform(seed + 2, (spec.K,), -0.1, 0.1)
    elif dist == "normal":
        x = _normal(seed, xs, 1.0)
        w = _normal(seed + 1, ws, math.sqrt(1.0 / crs))
        bias = _uniform(seed + 2, (spec.K,), -0.1, 0.1)
    elif dist == "relu":
        x = np.maximum(_normal(seed, xs, 1.0), 0.0)
        w = _normal(seed + 1, ws, math.sqrt(2.0 / crs))
        bias = _uniform(seed + 2, (spec.K,), -0.1, 0.1)
    elif dist == "positive":
        x = _uniform(seed, xs, 0.0, 1.0)
        w = _uniform(seed + 1, ws, 0.0, 1.0)
        bias = _uniform(seed + 2, (spec.K,), 0.0, 1.0)
    else:
        raise ValueError(dist)
    b = _finish(bias, spec, "b") if spec.bias else None
    return _finish(x, spec, "x"), _finish(w, spec, "w"), b


def workload_inputs(spec: ConvSpec):
    """Inputs of any named workload above, by its documented recipe."""
    if spec == MSCRED_SINGLE:
        return mscred_single_inputs(spec)
    if spec == CNN_MID_F16:
        return layer_inputs(spec, 2, 0, "mid")
    for i, s in enumerate(KSWEEP_BF16):
        if spec == s:
            return layer_inputs(spec, 3, i, "normal")
    for i, s in enumerate(DEEP_BF16):
        if spec == s:
            return layer_inputs(spec, 4, i, "relu")
    for i, s in enumerate(MSCRED_ENCODER):
        if spec == s:
            w, b = kaiming_params(spec, 1000 + 10 * i)
            x = layer_inputs(spec, 1, i, "normal")[0]
            return x, w, b
    raise KeyError(spec.name)


TENSOR_CORE_WORKLOADS: List[ConvSpec] = [CNN_MID_F16] + KSWEEP_BF16 + DEEP_BF16
ALL_LAYERS: Dict[str, ConvSpec] = {s.name: s for s in
                                   [MSCRED_SINGLE] + MSCRED_ENCODER + TENSOR_CORE_WORKLOADS}


def random_spec(rng: np.random.Generator, dtype: str, layout: str, max_dim: int = 20) -> ConvSpec:
    """A small random layer with a valid (non-empty) output, for parity sweeps."""
    while True:
        R = int(rng.integers(1, 6))
        S = int(rng.integers(1, 6))
        st = int(rng.integers(1, 4))
        dil = int(rng.integers(1, 3))
        pad = int(rng.integers(0, 4))
        H = int(rng.integers(1, max_dim))
        W = int(rng.integers(1, max_dim))
        if H + 2 * pad - dil * (R - 1) - 1 < 0 or W + 2 * pad - dil * (S - 1) - 1 < 0:
            continue
        C = int(rng.integers(1, 40))
        K = int(rng.integers(1, 40))
        N = int(rng.integers(1, 4))
        return ConvSpec(f"rand_{dtype}_{layout}", N, C, H, W, K, R, S, st, pad, dil,
                        dtype=dtype, layout=layout, bias=bool(rng.integers(0, 2)))


def random_inputs(spec: ConvSpec, seed: int, dist: str = "normal"):
    crs = spec.C * spec.R * spec.S
    xs = (spec.N, spec.C, spec.H, spec.W)
    ws = (spec.K, spec.C, spec.R, spec.S)
    if dist == "positive":
        x = _uniform(seed, xs, 0.0, 1.0)
        w = _uniform(seed + 1, ws, 0.0, 1.0)
        bias = _uniform(seed + 2, (spec.K,), 0.0, 1.0)
    else:
        x = _normal(seed, xs, 1.0)
        w = _normal(seed + 1, ws, math.sqrt(1.0 / crs))
        bias = _uniform(seed + 2, (spec.K,), -0.5, 0.5)
    b = _finish(bias, spec, "b") if spec.bias else None
    return _finish(x, spec, "x"), _finish(w, spec, "w"), b


# ------------------------------------------------------------ output sample points
#
# Where a whole output is too large to check against the oracle, these pick
# the logical outputs (n, k, p, q) to check.  Index selection only.

def sample_indices(spec: ConvSpec, P: int, Q: int, count: int, seed: int) -> np.ndarray:
    """Random outputs plus every border pixel of the first and last image
    (8 random channels)."""
    rng = np.random.default_rng(seed)
    idx = [np.stack([rng.integers(0, d, size=count) for d in (spec.N, spec.K, P, Q)], axis=1)]
    ks = rng.integers(0, spec.K, size=min(spec.K, 8))
    for n in sorted({0, spec.N - 1}):
        for k in ks:
            for p in range(P):
                for q in range(Q):
                    if p in (0, P - 1) or q in (0, Q - 1):
                        idx.append(np.array([[n, k, p, q]]))
    return np.concatenate(idx, axis=0)


def stratified_indices(spec: ConvSpec, P: int, Q: int, seed: int, tile_m: int = 128,
                       chunk_k: int = 32) -> np.ndarray:
    """Outputs that put at least two checked points into every output tile.

    The GEMM rows m = (n, p, q) are cut into blocks of tile_m (the kernels'
    M tile); for each block its first and last row are checked.  Window-mode
    tiles are whole output rows, so the first and last pixel of every output
    row are checked too.  Each such pixel is paired with one random channel
    of every chunk_k-channel group (the epilogue's store box), so every
    (M tile, N tile) and every store of a tile has checked elements."""
    rng = np.random.default_rng(seed)
    M = spec.N * P * Q
    firsts = np.arange(0, M, tile_m, dtype=np.int64)
    lasts = np.minimum(firsts + tile_m, M) - 1
    row_starts = np.arange(spec.N * P, dtype=np.int64) * Q
    rows = np.unique(np.concatenate([firsts, lasts, row_starts, row_starts + Q - 1]))
    n, rem = np.divmod(rows, P * Q)
    p, q = np.divmod(rem, Q)
    out = []
    for k0 in range(0, spec.K, chunk_k):
        k = rng.integers(k0, min(k0 + chunk_k, spec.K), size=rows.size)
        out.append(np.stack([n, k, p, q], axis=1))
    return np.concatenate(out, axis=0)


def check_points(spec: ConvSpec, P: int, Q: int, seed: int = 0, count: int = 6000) -> np.ndarray:
    """Random, border and stratified sample points of one layer's output."""
    return np.concatenate([sample_indices(spec, P, Q, count, seed),
                           stratified_indices(spec, P, Q, seed + 1)], axis=0)


def gather_points(y: torch.Tensor, idx: np.ndarray, layout: str) -> torch.Tensor:
    """y at logical outputs idx[i] = (n, k, p, q), on y's device."""
    t = torch.as_tensor(idx, dtype=torch.long, device=y.device)
    n, k, p, q = t.unbind(1)
    return y[n, k, p, q] if layout == "NCHW" else y[n, p, q, k]
