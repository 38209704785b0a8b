"""Seeded synthetic workloads for the W4A4 NVFP4 quantised projection.

This module is the ONLY code shared by the CUDA path's tests/benchmarks and the
CPU oracle.  It draws inputs (activations x, weights W, bias b) and the offline
calibration products that the method treats as inputs (smoothing vector s,
outlier index set Omega, low-rank factors L1/L2).  It contains none of the
hot-path arithmetic (no Walsh-Hadamard transform, no NVFP4 rounding, no
folding, no GEMM): those live independently in ``oracle/`` and in the CUDA
library.

Workload shapes follow the deployment scenarios of the pages:
  * "tiny"      — a single projection, M=8, K=256 -> N=512, four outlier channels x30,
                  rank-16 low-rank branch (QuantWAMs Fig. 1 style outliers).
  * "expert"    — action-expert projections at batch 1 (FoldQuantVLA, sec. "What This
                  Paper Is About": latency-critical batch-1 expert), M=50 tokens,
                  up 1024->4096 and down 4096->1024, rank 32, eight outlier channels x20.
  * "backbone"  — language-backbone prefill, M=768, QKV/gate-up in W4A4, o_proj and
                  down_proj in W8A8 (FoldQuantVLA, Key Contribution 3), Student-t(4)
                  activations with 16 outlier channels x50.
  * "video_dit" — a video DiT block, M=16384, log-normal per-channel magnitudes,
                  rank 32 plus the top-64 pooled-squared-energy channels kept in FP16
                  (QuantWAMs sec. 3.1, Eq. (1)-(3)).
  * "vae_conv"  — a Wan-style VAE 3x3x3 Conv3d, C=384, 1x384x5x60x104 (LatentQuant
                  abstract: NVFP4 execution of the video VAE).

Calibration products (offline, per the pages they are computed before deployment):
  * s_j = sqrt(max_m |x_mj| / max_n |W_jn|)  (SmoothQuant alpha = 0.5, the smoothing
    the pages take as a baseline/ingredient; s_j = 1 where either max is 0).
  * L1, L2 = top-r SVD factors of diag(s) W  (SVDQuant-style, a baseline the pages compare
    against; Q-WAM's "tiny 16-bit low-rank branch").
  * Omega = Top-K of the pooled squared energy z(c) = mean_t xt[t,c]^2 of the
    transformed input xt = (x diag(s)^-1) H (QuantWAMs sec. 3.1 Eq. (1)-(3), one context,
    pi = 1).  H is applied here as a dense block-diagonal Sylvester matrix from scipy,
    only to rank channels; ties broken by the lower index; Omega sorted ascending.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

__all__ = ["LayerSpec", "Workload", "WORKLOADS", "make_layer_inputs", "bf16_round",
           "bf16_bits", "bf16_from_bits", "outlier_channels", "make_conv_inputs"]


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    name: str
    K: int
    N: int
    mode: str = "w4a4"        # "w4a4" or "w8a8"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    layers: tuple
    dist: str                 # "gauss", "student_t4", "lognormal_channels"
    n_outlier_ch: int         # planted outlier channels
    outlier_mult: float
    rank: int
    n_omega: int              # |Omega| kept in fp16
    bias: bool
    rotate: bool
    smooth: bool
    seed: int
    x_fp32_source: bool = False   # inputs drawn as fp32 and rounded to bf16 at the boundary


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 8, (LayerSpec("proj", 256, 512),), "gauss", 4, 30.0,
                     rank=16, n_omega=0, bias=False, rotate=True, smooth=True, seed=0,
                     x_fp32_source=True),
    "expert": Workload("expert", 50, (LayerSpec("up", 1024, 4096), LayerSpec("down", 4096, 1024)),
                       "gauss", 8, 20.0, rank=32, n_omega=0, bias=True, rotate=True,
                       smooth=True, seed=1),
    "backbone": Workload("backbone", 768,
                         (LayerSpec("qkv", 2048, 6144), LayerSpec("o_proj", 2048, 2048, "w8a8"),
                          LayerSpec("gate_up", 2048, 32768), LayerSpec("down", 16384, 2048, "w8a8")),
                         "student_t4", 16, 50.0, rank=0, n_omega=0, bias=True, rotate=True,
                         smooth=True, seed=2),
    "video_dit": Workload("video_dit", 16384,
                          (LayerSpec("qkv", 1536, 4608), LayerSpec("o", 1536, 1536),
                           LayerSpec("up", 1536, 8960), LayerSpec("down", 8960, 1536)),
                          "lognormal_channels", 0, 1.0, rank=32, n_omega=64, bias=True,
                          rotate=True, smooth=True, seed=3),
}

CONV = dict(name="vae_conv", C_in=384, C_out=384, T=5, H=60, W=104, k=3, pad=1,
            n_outlier_ch=6, outlier_mult=25.0, seed=4)


# ---------------------------------------------------------------- bf16 helpers
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 -> bf16 (round to nearest even) and return the uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(a: np.ndarray) -> np.ndarray:
    return bf16_from_bits(bf16_bits(a))


# ---------------------------------------------------------------- generators
def outlier_channels(K: int, n: int) -> np.ndarray:
    """Evenly spaced planted outlier channels j_i = floor((i + 1/2) K / n)."""
    return np.array([int((i + 0.5) * K / n) for i in range(n)], dtype=np.int64)


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, *stream])


def _draw_x(wl: Workload, M: int, K: int, layer_idx: int, rows: Optional[np.ndarray] = None) -> np.ndarray:
    g = _rng(wl.seed, layer_idx, 1)
    if wl.dist == "gauss":
        x = g.standard_normal((M, K), dtype=np.float32)
    elif wl.dist == "student_t4":
        z = g.standard_normal((M, K), dtype=np.float32)
        chi = g.chisquare(4.0, size=(M, K)).astype(np.float32)
        x = z / np.sqrt(chi / 4.0)
    elif wl.dist == "lognormal_channels":
        c = np.exp(_rng(wl.seed, layer_idx, 2).standard_normal(K)).astype(np.float32)
        x = g.standard_normal((M, K), dtype=np.float32) * c[None, :]
    else:
        raise ValueError(wl.dist)
    if wl.n_outlier_ch:
        x[:, outlier_channels(K, wl.n_outlier_ch)] *= np.float32(wl.outlier_mult)
    return x


def _draw_w(wl: Workload, K: int, N: int, layer_idx: int) -> np.ndarray:
    return (_rng(wl.seed, layer_idx, 3).standard_normal((K, N), dtype=np.float32)
            * np.float32(0.02))


def _draw_b(wl: Workload, N: int, layer_idx: int) -> Optional[np.ndarray]:
    if not wl.bias:
        return None
    return _rng(wl.seed, layer_idx, 4).standard_normal(N, dtype=np.float32) * np.float32(0.02)


def smoothing_factors(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    ax = np.abs(x).max(axis=0).astype(np.float64)
    aw = np.abs(W).max(axis=1).astype(np.float64)
    s = np.ones(x.shape[1], dtype=np.float64)
    ok = (ax > 0) & (aw > 0)
    s[ok] = np.sqrt(ax[ok] / aw[ok])
    return s.astype(np.float32)


def lowrank_factors(W: np.ndarray, s: np.ndarray, r: int):
    if r == 0:
        return None, None
    Ws = W.astype(np.float64) * s.astype(np.float64)[:, None]
    U, S, Vt = np.linalg.svd(Ws, full_matrices=False)
    L1 = (U[:, :r] * S[None, :r]).astype(np.float32)
    L2 = Vt[:r, :].astype(np.float32)
    return L1, L2


def _block_hadamard(a: np.ndarray, axis: int) -> np.ndarray:
    """Dense block-64 Sylvester transform (1/8 normalised) along `axis`, fp64 (calibration only)."""
    from scipy.linalg import hadamard
    H = hadamard(64).astype(np.float64) / 8.0
    a = np.moveaxis(np.asarray(a, np.float64), axis, -1)
    sh = a.shape
    out = (a.reshape(*sh[:-1], sh[-1] // 64, 64) @ H).reshape(sh)
    return np.moveaxis(out, -1, axis)


def pooled_energy_topk(x: np.ndarray, s: np.ndarray, k_out: int, rotate: bool,
                       smooth_after: bool = False) -> np.ndarray:
    """Top-K channels of z(c) = mean_t xt[t,c]^2 on the transformed input (dense H)."""
    if k_out == 0:
        return np.zeros(0, dtype=np.int32)
    M, K = x.shape
    z = np.zeros(K, dtype=np.float64)
    step = 2048
    for m0 in range(0, M, step):
        xs = x[m0:m0 + step].astype(np.float64)
        if smooth_after and rotate:
            xs = _block_hadamard(xs, 1) / s.astype(np.float64)[None, :]
        else:
            xs = xs / s.astype(np.float64)[None, :]
            if rotate:
                xs = _block_hadamard(xs, 1)
        z += (xs * xs).sum(axis=0)
    z /= M
    order = sorted(range(K), key=lambda c: (-z[c], c))[:k_out]
    return np.array(sorted(order), dtype=np.int32)


@dataclasses.dataclass
class LayerInputs:
    wl: Workload
    spec: LayerSpec
    M: int
    x_bits: np.ndarray            # uint16 [M, K] bf16 bit patterns
    W: np.ndarray                 # fp32 [K, N]
    bias: Optional[np.ndarray]    # fp32 [N] or None
    s: Optional[np.ndarray]       # fp32 [K] or None
    L1: Optional[np.ndarray]      # fp32 [K, r]
    L2: Optional[np.ndarray]      # fp32 [r, N]
    omega: np.ndarray             # int32 [n_omega]
    rotate: bool = True
    smooth_after: bool = False    # rotation first, then smoothing (QuantWAMs Eq. (1))

    @property
    def x_f32(self) -> np.ndarray:
        return bf16_from_bits(self.x_bits)

    @property
    def rank(self) -> int:
        return 0 if self.L1 is None else self.L1.shape[1]


def make_layer_inputs(workload: str, layer: int = 0, M: Optional[int] = None,
                      K: Optional[int] = None, N: Optional[int] = None,
                      rank: Optional[int] = None, n_omega: Optional[int] = None,
                      smooth: Optional[bool] = None, rotate: Optional[bool] = None,
                      smooth_after: bool = False) -> LayerInputs:
    """Draw one layer of a workload.  Shape/feature overrides give smaller parity cases
    with the same distributions (the seed stream is unchanged).  smooth_after: the
    calibration products are taken in the rotate-then-smooth basis (s from the rotated
    activations and weights, the low-rank factors of S H W, Omega of x H S^-1)."""
    wl = WORKLOADS[workload]
    spec = wl.layers[layer]
    M = wl.M if M is None else M
    K = spec.K if K is None else K
    N = spec.N if N is None else N
    r = wl.rank if rank is None else rank
    n_om = wl.n_omega if n_omega is None else n_omega
    do_smooth = wl.smooth if smooth is None else smooth
    do_rot = wl.rotate if rotate is None else rotate
    x = _draw_x(wl, M, K, layer)
    x_bits = bf16_bits(x)
    xb = bf16_from_bits(x_bits)
    W = _draw_w(wl, K, N, layer)
    b = _draw_b(wl, N, layer)
    after = bool(smooth_after) and do_rot
    if after:
        xr = _block_hadamard(xb, 1).astype(np.float32)          # x H
        Wr = _block_hadamard(W, 0).astype(np.float32)           # H W (H symmetric)
        s = smoothing_factors(xr, Wr) if do_smooth else None
        s_eff = s if s is not None else np.ones(K, dtype=np.float32)
        L1, L2 = lowrank_factors(Wr, s_eff, r) if (spec.mode == "w4a4" and r > 0) else (None, None)
    else:
        s = smoothing_factors(xb, W) if do_smooth else None
        s_eff = s if s is not None else np.ones(K, dtype=np.float32)
        L1, L2 = lowrank_factors(W, s_eff, r) if (spec.mode == "w4a4" and r > 0) else (None, None)
    omega = pooled_energy_topk(xb, s_eff, n_om, do_rot, after) if spec.mode == "w4a4" else np.zeros(0, np.int32)
    return LayerInputs(wl, dataclasses.replace(spec, K=K, N=N), M, x_bits, W, b, s, L1, L2, omega, do_rot, after)


def make_conv_inputs(T: Optional[int] = None, H: Optional[int] = None, W: Optional[int] = None,
                     C_in: Optional[int] = None, C_out: Optional[int] = None, B: int = 1):
    """VAE Conv3d input (NCDHW bf16 bits, batch B) and weights [C_out, C_in, 3, 3, 3] fp32."""
    c = dict(CONV)
    T = c["T"] if T is None else T
    H = c["H"] if H is None else H
    W_ = c["W"] if W is None else W
    Ci = c["C_in"] if C_in is None else C_in
    Co = c["C_out"] if C_out is None else C_out
    g = _rng(c["seed"], 0, 1)
    x = g.standard_normal((B, Ci, T, H, W_), dtype=np.float32)
    x[:, outlier_channels(Ci, c["n_outlier_ch"])] *= np.float32(c["outlier_mult"])
    w = _rng(c["seed"], 0, 3).standard_normal((Co, Ci, 3, 3, 3), dtype=np.float32) * np.float32(0.02)
    return bf16_bits(x), w
