"""CPU oracle for the W4A4 NVFP4 quantised projection -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and this
package never imports the product library.  The arithmetic is in ``oracle.c``
(plain C, fp64 accumulation, fixed-order fp32 transforms); this file only
compiles it with gcc and marshals numpy arrays through ctypes.

Every function states the passage it follows in ``oracle.c``'s header.
Parity pins live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i64, i32, f32 = ctypes.c_long, ctypes.c_int, ctypes.c_float
            L.orc_e2m1_encode.argtypes = [f32]; L.orc_e2m1_encode.restype = ctypes.c_uint8
            L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]; L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e4m3_encode.argtypes = [f32]; L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]; L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_bf16_from_f64.argtypes = [ctypes.c_double]; L.orc_bf16_from_f64.restype = ctypes.c_uint16
            L.orc_fwht64_f32.argtypes = [P]; L.orc_fwht64_f32.restype = None
            L.orc_fwht64_f64.argtypes = [P, i64]; L.orc_fwht64_f64.restype = None
            L.orc_nvfp4_quantize.argtypes = [P, i64, f32, P, P]; L.orc_nvfp4_quantize.restype = None
            L.orc_quantize_act.argtypes = [P, i64, i64, P, i32, P, i32, i32, P, P, P, P, P, i32]
            L.orc_quantize_act.restype = i32
            L.orc_fold_weights.argtypes = [P, i64, i64, P, P, P, i32, P, i32, i32, P, P, P, P, P, i32]
            L.orc_fold_weights.restype = i32
            L.orc_quantize_weights.argtypes = [P, i64, i64, P, P, P]; L.orc_quantize_weights.restype = i32
            L.orc_lowrank_act.argtypes = [P, i64, i64, P, i32, P]; L.orc_lowrank_act.restype = None
            L.orc_linear_forward.argtypes = [P, P, P, i32, i64, P, P, f32, i64, i64, P, P, i32,
                                             P, P, i32, P, P, i32]
            L.orc_linear_forward.restype = i32
            L.orc_forward_noquant.argtypes = [P, P, i64, i64, i64, P, P, i32, P, P, P, i32, P, P]
            L.orc_forward_noquant.restype = i32
            L.orc_conv3d_forward.argtypes = [P, P, f32, i64, i64, i64, i64, P, P, f32, i64, P, i64, P, i32]
            L.orc_conv3d_forward.restype = i32
            L.orc_quantize_act_int8.argtypes = [P, i64, i64, P, i32, P, P, i32]
            L.orc_quantize_act_int8.restype = i32
            L.orc_quantize_weights_int8.argtypes = [P, i64, i64, P, P]
            L.orc_quantize_weights_int8.restype = i32
            L.orc_linear_forward_w8a8.argtypes = [P, P, i64, P, P, i64, i64, P, P, i32]
            L.orc_linear_forward_w8a8.restype = i32
            L.orc_set_smooth_after.argtypes = [i32]
            L.orc_set_smooth_after.restype = None
            L.orc_pooled_energy.argtypes = [P, i64, i64, P, i32, P]; L.orc_pooled_energy.restype = i32
            L.orc_projection_basis.argtypes = [P, i64, i32, i32, P]; L.orc_projection_basis.restype = i32
            L.orc_project_complement.argtypes = [P, i64, i64, P, P, i32]; L.orc_project_complement.restype = None
            L.orc_quantize_act_projected.argtypes = [P, i64, i64, P, i32, P, i32, P, P, i32, P, P, P, P, P]
            L.orc_quantize_act_projected.restype = i32
            L.orc_topk_channels.argtypes = [P, i64, i32, P]; L.orc_topk_channels.restype = i32
            L.orc_e4m3s_encode.argtypes = [f32]; L.orc_e4m3s_encode.restype = ctypes.c_uint8
            L.orc_e4m3s_decode.argtypes = [ctypes.c_uint8]; L.orc_e4m3s_decode.restype = ctypes.c_double
            L.orc_quantize_act_fp8.argtypes = [P, i64, i64, P, i32, P, i32, P, P, P, i32]
            L.orc_quantize_act_fp8.restype = i32
            L.orc_quantize_weights_fp8.argtypes = [P, i64, i64, P, P]
            L.orc_quantize_weights_fp8.restype = i32
            L.orc_linear_forward_fp8.argtypes = [P, P, i64, P, P, i64, i64, P, P, i32]
            L.orc_linear_forward_fp8.restype = i32
            L.orc_linear_forward_w4a8.argtypes = [P, P, i64, P, P, f32, i64, i64, P, P, i32, P, P, i32, P, P, i32]
            L.orc_linear_forward_w4a8.restype = i32
            _lib = L
    return _lib


_order_lock = threading.RLock()


class transform_order:
    """Context for the transform order of the oracle calls made inside it: smooth_after=False is
    smoothing then rotation (FoldQuantVLA, Key Contribution 2), True is rotation then smoothing
    (QuantWAMs sec. 3.1 Eq. (1), A R S^-1)."""

    def __init__(self, smooth_after: bool):
        self.v = bool(smooth_after)

    def __enter__(self):
        _order_lock.acquire()
        lib().orc_set_smooth_after(int(self.v))
        return self

    def __exit__(self, *a):
        lib().orc_set_smooth_after(0)
        _order_lock.release()


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ scalar formats
def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(v)))


def e2m1_decode(c: int) -> float:
    return float(lib().orc_e2m1_decode(int(c)))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e4m3_decode(c: int) -> float:
    return float(lib().orc_e4m3_decode(int(c)))


def fwht64_f32(v: np.ndarray) -> np.ndarray:
    """FoldQuantVLA Key Contribution 2: block Hadamard by FWHT, beta = 64 (fp32)."""
    out = np.array(v, dtype=np.float32, copy=True)
    assert out.shape == (64,)
    lib().orc_fwht64_f32(_p(out))
    return out


def fwht64_f64(v: np.ndarray) -> np.ndarray:
    out = np.array(v, dtype=np.float64, copy=True)
    assert out.shape == (64,)
    lib().orc_fwht64_f64(_p(out), 1)
    return out


def nvfp4_quantize(v: np.ndarray, g: float):
    """NVFP4 two-level quantisation of a vector with a given fp32 tensor scale g."""
    v = _c(v, np.float32)
    n = v.size
    codes = np.zeros(n // 2, np.uint8)
    scales = np.zeros(n // 16, np.uint8)
    lib().orc_nvfp4_quantize(_p(v), n, np.float32(g), _p(codes), _p(scales))
    return codes, scales


def inv_smoothing(s: Optional[np.ndarray]) -> Optional[np.ndarray]:
    """inv_s = 1/s, one IEEE fp32 division per channel."""
    if s is None:
        return None
    s = np.asarray(s, np.float32)
    return (np.float32(1.0) / s).astype(np.float32)


# ------------------------------------------------------------------ activations
@dataclass
class ActQuant:
    codes: np.ndarray        # uint8 [M, K/2], element 2i in the low nibble
    scales: np.ndarray       # uint8 [M, K/16] (e4m3)
    g: np.ndarray            # fp32 [M] (per row) or [1] (per tensor)
    x_omega: np.ndarray      # fp16 bits [M, n_omega]
    xt: Optional[np.ndarray] = None   # fp32 [M, K] transformed rows, outliers zeroed


def quantize_act(x_bits: np.ndarray, s: Optional[np.ndarray], rotate: bool,
                 omega: Optional[np.ndarray] = None, per_tensor: bool = False,
                 keep_xt: bool = False, n_threads: int = 0, static_g: Optional[float] = None) -> ActQuant:
    """Smoothing -> block FWHT -> outlier split -> NVFP4 (FoldQuantVLA contribution 2;
    QuantWAMs sec. 3.1 Eq. (1)).  Tensor scale: per row (default), one per batch from its
    amax (per_tensor), or a fixed calibrated g (static_g)."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    inv_s = inv_smoothing(s)
    omega = np.zeros(0, np.int32) if omega is None else _c(omega, np.int32)
    no = int(omega.size)
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    g = np.zeros(1 if (per_tensor or static_g is not None) else M, np.float32)
    mode = 0
    if static_g is not None:
        g[0] = np.float32(static_g)
        mode = 2
    elif per_tensor:
        mode = 1
    xo = np.zeros((M, no), np.uint16)
    xt = np.zeros((M, K), np.float32) if keep_xt else None
    rc = lib().orc_quantize_act(_p(x_bits), M, K, _p(inv_s), int(rotate), _p(omega), no,
                                mode, _p(codes), _p(scales), _p(g), _p(xo), _p(xt),
                                int(n_threads))
    if rc:
        raise ValueError(f"orc_quantize_act failed: {rc}")
    return ActQuant(codes, scales, g, xo, xt)


# ------------------------------------------------------------------ weights
@dataclass
class WeightQuant:
    codes: np.ndarray        # uint8 [N, K/2]
    scales: np.ndarray       # uint8 [N, K/16]
    gW: float
    W_omega: np.ndarray      # fp16 bits [n_omega, N]
    P: np.ndarray            # bf16 bits [K, r]
    Q: np.ndarray            # bf16 bits [r, N]
    Rp: np.ndarray           # fp32 [K, N] folded weight (outlier rows zeroed)
    W_omega_f32: np.ndarray  # fp32 [n_omega, N]


def prepare_weights(W: np.ndarray, s: Optional[np.ndarray], L1: Optional[np.ndarray],
                    L2: Optional[np.ndarray], omega: Optional[np.ndarray], rotate: bool,
                    n_threads: int = 0) -> WeightQuant:
    """Consistent folding (FoldQuantVLA Prop. 1) of smoothing + rotation into W, the
    16-bit low-rank complement (Q-WAM ASP), the fp16 outlier rows (QuantWAMs sec. 3.1),
    then per-tensor NVFP4 of the folded weight."""
    W = _c(W, np.float32)
    K, N = W.shape
    r = 0 if L1 is None else L1.shape[1]
    s = _c(s, np.float32)
    L1 = _c(L1, np.float32)
    L2 = _c(L2, np.float32)
    omega = np.zeros(0, np.int32) if omega is None else _c(omega, np.int32)
    no = int(omega.size)
    Rp = np.zeros((K, N), np.float32)
    Wo = np.zeros((no, N), np.uint16)
    Wo32 = np.zeros((no, N), np.float32)
    P = np.zeros((K, r), np.uint16)
    Q = np.zeros((r, N), np.uint16)
    rc = lib().orc_fold_weights(_p(W), K, N, _p(s), _p(L1), _p(L2), r, _p(omega), no,
                                int(rotate), _p(Rp), _p(Wo), _p(Wo32), _p(P), _p(Q), int(n_threads))
    if rc:
        raise ValueError(f"orc_fold_weights failed: {rc}")
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    gW = np.zeros(1, np.float32)
    rc = lib().orc_quantize_weights(_p(Rp), K, N, _p(codes), _p(scales), _p(gW))
    if rc:
        raise ValueError(f"orc_quantize_weights failed: {rc}")
    return WeightQuant(codes, scales, float(gW[0]), Wo, P, Q, Rp, Wo32)


def lowrank_act(x_bits: np.ndarray, P: np.ndarray) -> np.ndarray:
    """U = bf16(x P), the 16-bit low-rank down-projection (Q-WAM ASP)."""
    x_bits = _c(x_bits, np.uint16)
    P = _c(P, np.uint16)
    M, K = x_bits.shape
    r = P.shape[1]
    U = np.zeros((M, r), np.uint16)
    if r:
        lib().orc_lowrank_act(_p(x_bits), M, K, _p(P), r, _p(U))
    return U


def linear_forward(aq: ActQuant, wq: WeightQuant, U: Optional[np.ndarray],
                   bias: Optional[np.ndarray], per_tensor_act: bool = False,
                   n_threads: int = 0) -> np.ndarray:
    """y = gA gW (A4 . W4) + U Q + x_omega W_omega + b, accumulated in fp64."""
    M, K2 = aq.codes.shape
    K = 2 * K2
    N = wq.codes.shape[0]
    r = wq.P.shape[1]
    no = wq.W_omega.shape[0]
    y = np.zeros((M, N), np.float64)
    U = np.zeros((M, 0), np.uint16) if U is None else _c(U, np.uint16)
    bias = _c(bias, np.float32)
    rc = lib().orc_linear_forward(_p(aq.codes), _p(aq.scales), _p(aq.g), int(per_tensor_act), M,
                                  _p(wq.codes), _p(wq.scales), np.float32(wq.gW), N, K,
                                  _p(U), _p(wq.Q), r, _p(aq.x_omega), _p(wq.W_omega), no,
                                  _p(bias), _p(y), int(n_threads))
    if rc:
        raise ValueError(f"orc_linear_forward failed: {rc}")
    return y


def forward_noquant(x_bits, s, rotate, omega, wq: WeightQuant, bias, smooth_after: bool = False) -> np.ndarray:
    """The folded pipeline with quantisation disabled (FoldQuantVLA Proposition 1)."""
    with transform_order(smooth_after):
        return _forward_noquant(x_bits, s, rotate, omega, wq, bias)


def _forward_noquant(x_bits, s, rotate, omega, wq: WeightQuant, bias) -> np.ndarray:
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    N = wq.codes.shape[0]
    r = wq.P.shape[1]
    omega = np.zeros(0, np.int32) if omega is None else _c(omega, np.int32)
    no = omega.size
    aq = quantize_act(x_bits, s, rotate, omega, keep_xt=True)
    # unrounded transformed outlier values: recompute the rows without the split
    full = quantize_act(x_bits, s, rotate, None, keep_xt=True).xt
    xo = np.ascontiguousarray(full[:, omega]) if no else np.zeros((M, 0), np.float32)
    y = np.zeros((M, N), np.float64)
    bias = _c(bias, np.float32)
    lib().orc_forward_noquant(_p(aq.xt), _p(xo), M, K, N, _p(wq.Rp), _p(wq.W_omega_f32), no,
                              _p(x_bits), _p(wq.P), _p(wq.Q), r, _p(bias), _p(y))
    return y


def reference_forward(layer, n_threads: int = 0, rows: Optional[np.ndarray] = None):
    """Full oracle pass for one ``workloads`` layer: returns (y fp64, ActQuant, WeightQuant, U).
    ``rows`` restricts the activation side to a subset of rows (sampled parity)."""
    x_bits = layer.x_bits if rows is None else layer.x_bits[rows]
    rotate = layer.rotate
    with transform_order(getattr(layer, "smooth_after", False)):
        wq = prepare_weights(layer.W, layer.s, layer.L1, layer.L2, layer.omega, rotate, n_threads)
        aq = quantize_act(x_bits, layer.s, rotate, layer.omega, n_threads=n_threads)
    U = lowrank_act(x_bits, wq.P) if wq.P.shape[1] else None
    y = linear_forward(aq, wq, U, layer.bias, n_threads=n_threads)
    return y, aq, wq, U


def bf16_bits_from_f64(y: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of fp64 values, one rounding to nearest even each."""
    f = lib().orc_bf16_from_f64
    flat = np.ascontiguousarray(y, np.float64).reshape(-1)
    return np.array([f(float(v)) for v in flat], np.uint16).reshape(np.shape(y))


def chain_quantize(y: np.ndarray, s_next, rotate_next: bool, omega_next, g_next: float,
                   smooth_after: bool = False) -> ActQuant:
    """The next layer's quantised input from this layer's output (FoldQuantVLA Key Contribution 1:
    one basis per activation site, the consumer's transform applied where the input is made): the
    fp64 output rounded once to bf16 (the value a bf16 activation tensor holds), then the next
    layer's smoothing, rotation, kept-channel split and NVFP4 with its fixed tensor scale."""
    bits = bf16_bits_from_f64(y)
    with transform_order(smooth_after):
        return quantize_act(bits, s_next, rotate_next, omega_next, static_g=g_next)


# ------------------------------------------------------------------ W8A8
@dataclass
class Int8Quant:
    q: np.ndarray            # int8 [rows, K]
    scale: np.ndarray        # fp32 [rows]


def quantize_act_int8(x_bits, s, rotate, n_threads: int = 0) -> Int8Quant:
    """Symmetric per-token int8 of the transformed activations (FoldQuantVLA, Key
    Contribution 3: selective W8A8 in the shared basis)."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    inv_s = inv_smoothing(s)
    q = np.zeros((M, K), np.int8)
    a = np.zeros(M, np.float32)
    rc = lib().orc_quantize_act_int8(_p(x_bits), M, K, _p(inv_s), int(rotate), _p(q), _p(a), int(n_threads))
    if rc:
        raise ValueError(f"orc_quantize_act_int8 failed: {rc}")
    return Int8Quant(q, a)


def prepare_weights_int8(W, s, rotate, n_threads: int = 0) -> Int8Quant:
    """Fold smoothing + rotation into W (Proposition 1), then per-output-channel int8."""
    wq = prepare_weights(W, s, None, None, None, rotate, n_threads)
    K, N = wq.Rp.shape
    q = np.zeros((N, K), np.int8)
    w = np.zeros(N, np.float32)
    lib().orc_quantize_weights_int8(_p(np.ascontiguousarray(wq.Rp)), K, N, _p(q), _p(w))
    return Int8Quant(q, w)


def linear_forward_w8a8(aq: Int8Quant, wq8: Int8Quant, bias, n_threads: int = 0) -> np.ndarray:
    M, K = aq.q.shape
    N = wq8.q.shape[0]
    y = np.zeros((M, N), np.float64)
    bias = _c(bias, np.float32)
    lib().orc_linear_forward_w8a8(_p(aq.q), _p(aq.scale), M, _p(wq8.q), _p(wq8.scale), N, K, _p(bias), _p(y),
                                  int(n_threads))
    return y


def reference_forward_w8a8(layer, n_threads: int = 0, rows=None):
    x_bits = layer.x_bits if rows is None else layer.x_bits[rows]
    wq8 = prepare_weights_int8(layer.W, layer.s, layer.rotate, n_threads)
    aq = quantize_act_int8(x_bits, layer.s, layer.rotate, n_threads)
    return linear_forward_w8a8(aq, wq8, layer.bias, n_threads), aq, wq8


# ------------------------------------------------------------------ projected complement (Q-WAM ASP)
def projection_basis(L1: np.ndarray, rotate: bool) -> np.ndarray:
    """Vt = bf16(S_r^-2 L1^T H) [r, K]: the action subspace in the rotated basis, scaled so that
    u Vt (u = x P, the branch's down-projection) is the activation's component in it."""
    L1 = _c(L1, np.float32)
    K, r = L1.shape
    Vt = np.zeros((r, K), np.uint16)
    rc = lib().orc_projection_basis(_p(L1), K, r, int(rotate), _p(Vt))
    if rc:
        raise ValueError(f"orc_projection_basis failed: {rc}")
    return Vt


def quantize_act_projected(x_bits, s, rotate, omega, U, Vt, keep_xt: bool = False) -> ActQuant:
    """Q-WAM abstract: the activation quantiser on the complement of the protected subspace."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    inv_s = inv_smoothing(s)
    omega = np.zeros(0, np.int32) if omega is None else _c(omega, np.int32)
    no = int(omega.size)
    U = _c(U, np.uint16)
    Vt = _c(Vt, np.uint16)
    r = Vt.shape[0]
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    g = np.zeros(M, np.float32)
    xo = np.zeros((M, no), np.uint16)
    xt = np.zeros((M, K), np.float32) if keep_xt else None
    rc = lib().orc_quantize_act_projected(_p(x_bits), M, K, _p(inv_s), int(rotate), _p(omega), no, _p(U), _p(Vt), r,
                                          _p(codes), _p(scales), _p(g), _p(xo), _p(xt))
    if rc:
        raise ValueError(f"orc_quantize_act_projected failed: {rc}")
    return ActQuant(codes, scales, g, xo, xt)


def reference_forward_projected(layer, n_threads: int = 0, rows=None):
    """Full oracle pass of the projected-complement variant: (y fp64, ActQuant, WeightQuant, U, Vt)."""
    x_bits = layer.x_bits if rows is None else layer.x_bits[rows]
    wq = prepare_weights(layer.W, layer.s, layer.L1, layer.L2, layer.omega, layer.rotate, n_threads)
    U = lowrank_act(x_bits, wq.P)
    Vt = projection_basis(layer.L1, layer.rotate)
    aq = quantize_act_projected(x_bits, layer.s, layer.rotate, layer.omega, U, Vt)
    y = linear_forward(aq, wq, U, layer.bias, n_threads=n_threads)
    return y, aq, wq, U, Vt


# ------------------------------------------------------------------ outlier calibration
def pooled_energy(x_bits, s, rotate: bool, smooth_after: bool = False) -> np.ndarray:
    """z(c) = mean_t xt[t, c]^2 of the quantiser's transform (QuantWAMs sec. 3.1 Eq. (1)-(3),
    one context)."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    inv_s = inv_smoothing(s)
    z = np.zeros(K, np.float64)
    with transform_order(smooth_after):
        rc = lib().orc_pooled_energy(_p(x_bits), M, K, _p(inv_s), int(rotate), _p(z))
    if rc:
        raise ValueError(f"orc_pooled_energy failed: {rc}")
    return z


def topk_channels(z: np.ndarray, n: int) -> np.ndarray:
    """The n channels of largest z, ties to the lower index, ascending (QuantWAMs Eq. (3) Top-K)."""
    z = _c(z, np.float64)
    om = np.zeros(n, np.int32)
    rc = lib().orc_topk_channels(_p(z), z.size, int(n), _p(om))
    if rc:
        raise ValueError(f"orc_topk_channels failed: {rc}")
    return om


# ------------------------------------------------------------------ W8A8 in FP8
@dataclass
class Fp8Quant:
    q: np.ndarray            # uint8 e4m3 codes [rows, K]
    scale: np.ndarray        # fp32 [rows]
    x_omega: Optional[np.ndarray] = None   # fp16 bits [rows, n_omega] (kept channels)


def quantize_act_fp8(x_bits, s, rotate, n_threads: int = 0, omega=None) -> Fp8Quant:
    """Per-token e4m3 of the transformed activations (QuantWAMs sec. 4.2: FP8 W8A8 for the
    upgraded layers; A8 at the protected steps), scale = amax / 448; kept channels (omega) go to
    fp16 and are zeroed first."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    inv_s = inv_smoothing(s)
    omega = np.zeros(0, np.int32) if omega is None else _c(omega, np.int32)
    xo = np.zeros((M, omega.size), np.uint16)
    q = np.zeros((M, K), np.uint8)
    a = np.zeros(M, np.float32)
    rc = lib().orc_quantize_act_fp8(_p(x_bits), M, K, _p(inv_s), int(rotate), _p(omega), int(omega.size), _p(xo),
                                    _p(q), _p(a), int(n_threads))
    if rc:
        raise ValueError(f"orc_quantize_act_fp8 failed: {rc}")
    return Fp8Quant(q, a, xo)


def prepare_weights_fp8(W, s, rotate, n_threads: int = 0) -> Fp8Quant:
    """Fold smoothing + rotation into W (Proposition 1), then per-output-channel e4m3."""
    wq = prepare_weights(W, s, None, None, None, rotate, n_threads)
    K, N = wq.Rp.shape
    q = np.zeros((N, K), np.uint8)
    w = np.zeros(N, np.float32)
    lib().orc_quantize_weights_fp8(_p(np.ascontiguousarray(wq.Rp)), K, N, _p(q), _p(w))
    return Fp8Quant(q, w)


def linear_forward_fp8(aq: Fp8Quant, wq8: Fp8Quant, bias, n_threads: int = 0) -> np.ndarray:
    M, K = aq.q.shape
    N = wq8.q.shape[0]
    y = np.zeros((M, N), np.float64)
    bias = _c(bias, np.float32)
    lib().orc_linear_forward_fp8(_p(aq.q), _p(aq.scale), M, _p(wq8.q), _p(wq8.scale), N, K, _p(bias), _p(y),
                                 int(n_threads))
    return y


def reference_forward_fp8(layer, n_threads: int = 0, rows=None):
    x_bits = layer.x_bits if rows is None else layer.x_bits[rows]
    wq8 = prepare_weights_fp8(layer.W, layer.s, layer.rotate, n_threads)
    aq = quantize_act_fp8(x_bits, layer.s, layer.rotate, n_threads)
    return linear_forward_fp8(aq, wq8, layer.bias, n_threads), aq, wq8


def reference_forward_w4a8(layer, n_threads: int = 0, rows=None):
    """A W4 layer at an A8-protected step (QuantWAMs sec. 4.2, sec. 5): its NVFP4 weights, low-rank
    branch and kept channels, its activations in e4m3 per token.  Returns (y fp64, Fp8Quant,
    WeightQuant, U)."""
    x_bits = layer.x_bits if rows is None else layer.x_bits[rows]
    with transform_order(getattr(layer, "smooth_after", False)):
        wq = prepare_weights(layer.W, layer.s, layer.L1, layer.L2, layer.omega, layer.rotate, n_threads)
        aq = quantize_act_fp8(x_bits, layer.s, layer.rotate, n_threads, omega=layer.omega)
    U = lowrank_act(x_bits, wq.P) if wq.P.shape[1] else np.zeros((x_bits.shape[0], 0), np.uint16)
    M, K = aq.q.shape
    N = wq.codes.shape[0]
    r = wq.P.shape[1]
    no = wq.W_omega.shape[0]
    y = np.zeros((M, N), np.float64)
    bias = _c(layer.bias, np.float32)
    rc = lib().orc_linear_forward_w4a8(_p(aq.q), _p(aq.scale), M, _p(wq.codes), _p(wq.scales), np.float32(wq.gW), N,
                                       K, _p(_c(U, np.uint16)), _p(wq.Q), r, _p(aq.x_omega), _p(wq.W_omega), no,
                                       _p(bias), _p(y), int(n_threads))
    if rc:
        raise ValueError(f"orc_linear_forward_w4a8 failed: {rc}")
    return y, aq, wq, U


# ------------------------------------------------------------------ Conv3d (VAE)
def conv_weight_matrix(w: np.ndarray) -> np.ndarray:
    """[C_out, C_in, 3, 3, 3] -> W [K = (kd, kh, kw, c_in), N = C_out] (math y = x W)."""
    Co, Ci = w.shape[:2]
    return np.ascontiguousarray(np.transpose(w, (2, 3, 4, 1, 0)).reshape(27 * Ci, Co), dtype=np.float32)


def conv3d_reference(x_bits_ncdhw: np.ndarray, w: np.ndarray, vox: np.ndarray, n_threads: int = 0):
    """LatentQuant, Abstract (NVFP4 execution of the VAE): quantise the input once per voxel
    (one tensor scale over the whole [B, C, D, H, W] input), the weight per output channel along
    (kd, kh, kw, c_in), and convolve each sample's dequantised values directly with zero padding 1.
    vox indexes voxels over the batch, v = b D H W + (d H + h) W + w.  Returns (y [n_vox, C_out]
    fp64, activation ActQuant over all voxels, weight WeightQuant)."""
    B, C, D, H, W = x_bits_ncdhw.shape
    V1 = D * H * W
    xv = np.ascontiguousarray(x_bits_ncdhw.reshape(B, C, V1).transpose(0, 2, 1).reshape(B * V1, C))
    aq = quantize_act(xv, None, False, None, per_tensor=True, n_threads=n_threads)
    wq = prepare_weights(conv_weight_matrix(w), None, None, None, None, False, n_threads)
    vox = np.ascontiguousarray(vox, dtype=np.int64)
    N = w.shape[0]
    y = np.zeros((vox.size, N), np.float64)
    for b in range(B):
        sel = np.flatnonzero(vox // V1 == b)
        if sel.size == 0:
            continue
        local = np.ascontiguousarray(vox[sel] % V1, dtype=np.int64)
        codes = np.ascontiguousarray(aq.codes[b * V1:(b + 1) * V1])
        scales = np.ascontiguousarray(aq.scales[b * V1:(b + 1) * V1])
        yb = np.zeros((sel.size, N), np.float64)
        lib().orc_conv3d_forward(_p(codes), _p(scales), np.float32(aq.g[0]), C, D, H, W, _p(wq.codes),
                                 _p(wq.scales), np.float32(wq.gW), N, _p(local), local.size, _p(yb), int(n_threads))
        y[sel] = yb
    return y, aq, wq
