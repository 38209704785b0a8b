"""Python binding of libwq (include/wq.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; PyTorch provides device
memory and streams.  The functions keep the C names.  If ``libwq.so`` has not
been built, importing the binding's functions raises immediately: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")

WQ_OK, WQ_ERR_INVALID, WQ_ERR_UNSUPPORTED, WQ_ERR_CUDA, WQ_ERR_OOM, WQ_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
WQ_MODE_W4A4, WQ_MODE_W8A8, WQ_MODE_W8A8_FP8, WQ_MODE_W4A8 = 0, 1, 2, 3
WQ_SCALE_LAYOUT_ROWMAJOR, WQ_SCALE_LAYOUT_MMA = 0, 1
WQ_PATH_TWO_KERNEL, WQ_PATH_FUSED = 0, 1
WQ_GEMM_SINGLE, WQ_GEMM_SPLITK, WQ_GEMM_WIDE, WQ_GEMM_WIDE_DB = 0, 1, 2, 3
WQ_QUANT_CLUSTER, WQ_QUANT_STREAM, WQ_QUANT_RESIDENT = 0, 1, 2
WQ_ACT_SCALE_ROW, WQ_ACT_SCALE_TENSOR, WQ_ACT_SCALE_STATIC = 0, 1, 2
WQ_ORDER_SMOOTH_ROTATE, WQ_ORDER_ROTATE_SMOOTH = 0, 1

EXPORTED = ["wq_prepare_weights", "wq_get_config", "wq_workspace_bytes", "wq_linear_forward",
            "wq_host_workspace_bytes", "wq_linear_forward_host", "wq_quantize_activations",
            "wq_linear_forward_quantized", "wq_linear_forward_noalloc", "wq_linear_forward_w8a8",
            "wq_quantize_activations_w8a8", "wq_export_weights_w8a8", "wq_prepare_conv3d",
            "wq_conv3d_workspace_bytes", "wq_conv3d_forward", "wq_quantize_conv3d_input",
            "wq_export_weights", "wq_check_device_error", "wq_free_weights", "wq_last_error",
            "wq_forward_path", "wq_selftest_wait_timeout", "wq_gemm_schedule",
            "wq_quant_schedule", "wq_side_strides", "wq_set_tuning", "wq_get_tuning", "wq_mma_peak",
            "wq_linear_forward_chain", "wq_calibration_workspace_bytes", "wq_calibrate_outliers"]


class WqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"wq status {status}: {msg}")
        self.status = status


class wq_config(ctypes.Structure):
    _fields_ = [("K", ctypes.c_int), ("N", ctypes.c_int), ("rank", ctypes.c_int),
                ("n_outliers", ctypes.c_int), ("rotate", ctypes.c_int), ("mode", ctypes.c_int),
                ("act_scale", ctypes.c_int), ("act_gscale", ctypes.c_float), ("transform_order", ctypes.c_int),
                ("project", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libwq.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} not found: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.wq_prepare_weights.argtypes = [ctypes.POINTER(wq_config), P, P, P, P, P, P, P, ctypes.POINTER(P)]
        L.wq_prepare_weights.restype = I
        L.wq_get_config.argtypes = [P, ctypes.POINTER(wq_config)]
        L.wq_get_config.restype = I
        L.wq_side_strides.argtypes = [P, ctypes.POINTER(I), ctypes.POINTER(I)]
        L.wq_side_strides.restype = I
        L.wq_set_tuning.argtypes = [ctypes.c_char_p, I]
        L.wq_set_tuning.restype = I
        L.wq_get_tuning.argtypes = [ctypes.c_char_p]
        L.wq_get_tuning.restype = I
        L.wq_workspace_bytes.argtypes = [P, I]
        L.wq_workspace_bytes.restype = S
        L.wq_host_workspace_bytes.argtypes = [P, I]
        L.wq_host_workspace_bytes.restype = S
        L.wq_linear_forward.argtypes = [P, P, I, P, P, S, P]
        L.wq_linear_forward.restype = I
        L.wq_linear_forward_host.argtypes = [P, P, I, P, P, S, P]
        L.wq_linear_forward_host.restype = I
        L.wq_quantize_activations.argtypes = [P, P, I, I, P, P, P, P, P, P]
        L.wq_quantize_activations.restype = I
        L.wq_linear_forward_chain.argtypes = [P, P, P, I, P, P, P, P, P, S, P]
        L.wq_linear_forward_chain.restype = I
        L.wq_linear_forward_quantized.argtypes = [P, P, P, P, P, P, I, P, P]
        L.wq_linear_forward_quantized.restype = I
        L.wq_linear_forward_noalloc.argtypes = [P, P, I, P, P]
        L.wq_linear_forward_noalloc.restype = I
        L.wq_linear_forward_w8a8.argtypes = [P, P, I, P, P, S, P]
        L.wq_linear_forward_w8a8.restype = I
        L.wq_quantize_activations_w8a8.argtypes = [P, P, I, P, P, P]
        L.wq_quantize_activations_w8a8.restype = I
        L.wq_export_weights_w8a8.argtypes = [P, P, P]
        L.wq_export_weights_w8a8.restype = I
        L.wq_prepare_conv3d.argtypes = [P, I, I, I, I, I, I, P, ctypes.POINTER(P)]
        L.wq_prepare_conv3d.restype = I
        L.wq_conv3d_workspace_bytes.argtypes = [P, I, I, I, I]
        L.wq_conv3d_workspace_bytes.restype = S
        L.wq_conv3d_forward.argtypes = [P, P, I, I, I, I, P, P, S, P]
        L.wq_conv3d_forward.restype = I
        L.wq_quantize_conv3d_input.argtypes = [P, P, I, I, I, I, P, P, P, P, S, P]
        L.wq_quantize_conv3d_input.restype = I
        L.wq_export_weights.argtypes = [P, P, P, P, P, P, P]
        L.wq_export_weights.restype = I
        L.wq_check_device_error.argtypes = [P, P]
        L.wq_check_device_error.restype = I
        L.wq_forward_path.argtypes = [P, I]
        L.wq_forward_path.restype = I
        L.wq_gemm_schedule.argtypes = [P, I]
        L.wq_gemm_schedule.restype = I
        L.wq_quant_schedule.argtypes = [P, I]
        L.wq_quant_schedule.restype = I
        L.wq_selftest_wait_timeout.argtypes = [ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I)]
        L.wq_selftest_wait_timeout.restype = I
        D = ctypes.POINTER(ctypes.c_double)
        L.wq_mma_peak.argtypes = [I, I, I, I, I, I, I, I, I, D, D, D]
        L.wq_mma_peak.restype = I
        L.wq_calibration_workspace_bytes.argtypes = [I, I]
        L.wq_calibration_workspace_bytes.restype = S
        L.wq_calibrate_outliers.argtypes = [P, I, I, P, I, I, I, P, P, P, S, P]
        L.wq_calibrate_outliers.restype = I
        L.wq_free_weights.argtypes = [P]
        L.wq_free_weights.restype = None
        L.wq_last_error.argtypes = []
        L.wq_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def wq_last_error() -> str:
    return lib().wq_last_error().decode()


def _check(status: int):
    if status != WQ_OK:
        raise WqError(status, wq_last_error())


def _host(a, dtype):
    if a is None:
        return None, None
    arr = np.ascontiguousarray(a, dtype=dtype)
    return arr, arr.ctypes.data_as(ctypes.c_void_p)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class Weights:
    """Owner of a wq_weights_t handle."""
    handle: int
    cfg: wq_config

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.wq_free_weights(ctypes.c_void_p(self.handle))
            self.handle = None

    @property
    def K(self):
        return self.cfg.K

    @property
    def N(self):
        return self.cfg.N


def wq_prepare_weights(K: int, N: int, W, bias=None, s=None, L1=None, L2=None, omega=None,
                       rotate: bool = True, mode: int = WQ_MODE_W4A4, stream=None,
                       act_scale: int = WQ_ACT_SCALE_ROW, act_gscale: float = 0.0,
                       transform_order: int = WQ_ORDER_SMOOTH_ROTATE, project: bool = False) -> Weights:
    """Fold and quantise one projection (host inputs, numpy or CPU tensors).  project: quantise
    the activations' complement of the low-rank branch's subspace (Q-WAM ASP)."""
    rank = 0 if L1 is None else int(np.shape(L1)[1])
    n_out = 0 if omega is None else int(np.size(omega))
    cfg = wq_config(K, N, rank, n_out, int(bool(rotate)), mode, int(act_scale), float(act_gscale),
                    int(transform_order), int(bool(project)))
    keep = []
    ptrs = []
    for a, dt in ((W, np.float32), (bias, np.float32), (s, np.float32), (L1, np.float32),
                  (L2, np.float32), (omega, np.int32)):
        if a is not None and hasattr(a, "numpy"):
            a = a.detach().cpu().numpy()
        arr, p = _host(a, dt)
        keep.append(arr)
        ptrs.append(p)
    out = ctypes.c_void_p()
    _check(lib().wq_prepare_weights(ctypes.byref(cfg), *ptrs, ctypes.c_void_p(_stream_ptr(stream)),
                                    ctypes.byref(out)))
    return Weights(out.value, cfg)


def wq_get_config(w: Weights) -> wq_config:
    cfg = wq_config()
    _check(lib().wq_get_config(ctypes.c_void_p(w.handle), ctypes.byref(cfg)))
    return cfg


def wq_side_strides(w: Weights):
    """(u_ld, xo_ld): row strides of U and x_Omega in the quantiser's outputs."""
    u, xo = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().wq_side_strides(ctypes.c_void_p(w.handle), ctypes.byref(u), ctypes.byref(xo)))
    return u.value, xo.value


def wq_set_tuning(name: str, value: int):
    """Pin a schedule knob (tests and tuning); -1 / 0 restores the automatic choice."""
    _check(lib().wq_set_tuning(name.encode(), int(value)))


def wq_get_tuning(name: str) -> int:
    return int(lib().wq_get_tuning(name.encode()))


def wq_workspace_bytes(w: Weights, M: int) -> int:
    return int(lib().wq_workspace_bytes(ctypes.c_void_p(w.handle), int(M)))


def wq_host_workspace_bytes(w: Weights, M: int) -> int:
    return int(lib().wq_host_workspace_bytes(ctypes.c_void_p(w.handle), int(M)))


def _alloc_workspace(nbytes: int, device):
    import torch
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def wq_linear_forward(w: Weights, x, y=None, workspace=None, stream=None):
    """y[M, N] (bf16, device) = projection(x[M, K] bf16, device)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous() and x.shape[-1] == w.K
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, w.N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _alloc_workspace(wq_workspace_bytes(w, M), x.device)
    _check(lib().wq_linear_forward(ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), M,
                                   ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                                   workspace.numel(), ctypes.c_void_p(_stream_ptr(stream))))
    return y


NOALLOC_SCRATCH_BYTES = 16 << 20


def wq_linear_forward_noalloc(w: Weights, x, y, stream=None):
    """Forward for callers that cannot allocate: scratch is the library's static device
    array (NOALLOC_SCRATCH_BYTES); x and y are caller-owned device tensors."""
    _check(lib().wq_linear_forward_noalloc(ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), x.shape[0],
                                           ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(_stream_ptr(stream))))
    return y


def wq_linear_forward_host(w: Weights, x_host, y_host, workspace, stream=None):
    """End-to-end call on host (pinned) bf16 tensors; y_host is valid after the stream syncs."""
    M = x_host.shape[0]
    _check(lib().wq_linear_forward_host(ctypes.c_void_p(w.handle), ctypes.c_void_p(x_host.data_ptr()), M,
                                        ctypes.c_void_p(y_host.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                                        workspace.numel(), ctypes.c_void_p(_stream_ptr(stream))))
    return y_host


def wq_quantize_activations(w: Weights, x, scale_layout: int = WQ_SCALE_LAYOUT_ROWMAJOR, stream=None):
    """Run the activation quantiser alone; returns device tensors (codes, scales, g, x_omega, u);
    x_omega is [M, xo_ld] and u [M, u_ld] (wq_side_strides), zero beyond the configured counts."""
    import torch
    M, K = x.shape
    dev = x.device
    if w.cfg.mode == WQ_MODE_W4A8:
        codes = torch.empty((M, K), dtype=torch.bfloat16, device=dev)      # e4m3 values held as bf16
    else:
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    if scale_layout == WQ_SCALE_LAYOUT_MMA:
        scales = torch.zeros(((M + 127) // 128) * (K // 64) * 512, dtype=torch.uint8, device=dev)
    else:
        scales = torch.empty((M, K // 16), dtype=torch.uint8, device=dev)
    g = torch.empty(M, dtype=torch.float32, device=dev)
    u_ld, xo_ld = wq_side_strides(w)
    xo = torch.empty((M, xo_ld), dtype=torch.float16, device=dev) if w.cfg.n_outliers else None
    u = torch.empty((M, u_ld), dtype=torch.bfloat16, device=dev) if w.cfg.rank else None
    _check(lib().wq_quantize_activations(
        ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), M, int(scale_layout),
        ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(g.data_ptr()),
        ctypes.c_void_p(xo.data_ptr() if xo is not None else None),
        ctypes.c_void_p(u.data_ptr() if u is not None else None), ctypes.c_void_p(_stream_ptr(stream))))
    return codes, scales, g, xo, u


def wq_quantize_activations_into(w: Weights, x, codes, scales, g, x_omega=None, u=None,
                                 stream=None, scale_layout: int = WQ_SCALE_LAYOUT_MMA):
    """wq_quantize_activations into caller-owned device tensors."""
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else None)
    _check(lib().wq_quantize_activations(ctypes.c_void_p(w.handle), ptr(x), x.shape[0], int(scale_layout),
                                         ptr(codes), ptr(scales), ptr(g), ptr(x_omega), ptr(u),
                                         ctypes.c_void_p(_stream_ptr(stream))))


def wq_linear_forward_quantized(w: Weights, codes, scales_mma, g, u=None, x_omega=None, y=None, stream=None):
    """GEMM + epilogue on activations quantised with WQ_SCALE_LAYOUT_MMA (device tensors)."""
    import torch
    M = codes.shape[0]
    if y is None:
        y = torch.empty((M, w.N), dtype=torch.bfloat16, device=codes.device)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else None)
    _check(lib().wq_linear_forward_quantized(ctypes.c_void_p(w.handle), ptr(codes), ptr(scales_mma), ptr(g),
                                             ptr(u), ptr(x_omega), M, ptr(y), ctypes.c_void_p(_stream_ptr(stream))))
    return y


def wq_linear_forward_chain(w: Weights, w_next: Weights, x, workspace=None, stream=None):
    """Layer w on x, its output quantised in the GEMM epilogue for w_next: returns device
    tensors (codes [M, N/2], scales in the MMA layout, g [M], x_omega [M, xo_ld] or None) that
    wq_linear_forward_quantized(w_next, ...) consumes."""
    import torch
    M = x.shape[0]
    N = w.N
    dev = x.device
    codes = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
    scales = torch.zeros(((M + 127) // 128) * (N // 64) * 512, dtype=torch.uint8, device=dev)
    g = torch.empty(M, dtype=torch.float32, device=dev)
    _, xo_ld = wq_side_strides(w_next)
    xo = torch.empty((M, xo_ld), dtype=torch.float16, device=dev) if w_next.cfg.n_outliers else None
    if workspace is None:
        workspace = _alloc_workspace(wq_workspace_bytes(w, M), dev)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else None)
    _check(lib().wq_linear_forward_chain(ctypes.c_void_p(w.handle), ctypes.c_void_p(w_next.handle), ptr(x), M,
                                         ptr(codes), ptr(scales), ptr(g), ptr(xo), ptr(workspace), workspace.numel(),
                                         ctypes.c_void_p(_stream_ptr(stream))))
    return codes, scales, g, xo


def wq_export_weights(w: Weights) -> dict:
    """Prepared weights copied back to host in canonical layouts."""
    K, N, r, no = w.cfg.K, w.cfg.N, w.cfg.rank, w.cfg.n_outliers
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    gW = np.zeros(1, np.float32)
    P = np.zeros((K, r), np.uint16)
    Q = np.zeros((r, N), np.uint16)
    Wo = np.zeros((no, N), np.uint16)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(lib().wq_export_weights(ctypes.c_void_p(w.handle), vp(codes), vp(scales), vp(gW), vp(P), vp(Q), vp(Wo)))
    return dict(codes=codes, scales=scales, gW=float(gW[0]), P=P, Q=Q, W_omega=Wo)


def wq_forward_path(w: Weights, M: int) -> int:
    """WQ_PATH_TWO_KERNEL or WQ_PATH_FUSED: the path wq_linear_forward takes for M rows."""
    r = lib().wq_forward_path(ctypes.c_void_p(w.handle), M)
    if r < 0:
        _check(r)
    return r


def wq_gemm_schedule(w: Weights, M: int) -> int:
    """WQ_GEMM_SINGLE, WQ_GEMM_SPLITK, WQ_GEMM_WIDE or WQ_GEMM_WIDE_DB: the GEMM schedule for M rows."""
    r = lib().wq_gemm_schedule(ctypes.c_void_p(w.handle), M)
    if r < 0:
        _check(r)
    return r


def wq_quant_schedule(w: Weights, M: int) -> int:
    """WQ_QUANT_CLUSTER, WQ_QUANT_STREAM or WQ_QUANT_RESIDENT: the activation-quantiser schedule
    for M rows."""
    r = lib().wq_quant_schedule(ctypes.c_void_p(w.handle), M)
    if r < 0:
        _check(r)
    return r


def wq_selftest_wait_timeout():
    """Run the bounded-wait self-test; returns (status, site, waited_ms pair, released) without raising."""
    site, released = ctypes.c_int(0), ctypes.c_int(0)
    waited = (ctypes.c_double * 2)()
    st = lib().wq_selftest_wait_timeout(ctypes.byref(site), waited, ctypes.byref(released))
    return st, site.value, (waited[0], waited[1]), released.value


MMA_KIND = {"fp4": 0, "bf16": 1, "fp8": 2}


def wq_mma_peak(kind: str = "fp4", n: int = 256, pair: bool = False, copies: int = 0, copy_shape: int = 0,
                iters: int = 8192, feeder: int = 0, zero_data: bool = False, accs: int = 1):
    """Tensor-core issue-rate microbenchmark on the current device (synchronous): returns
    (TFLOP/s over all SMs, ns per MMA instruction, mean SM MHz during the run)."""
    t, ns, mhz = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(lib().wq_mma_peak(MMA_KIND[kind], n, int(bool(pair)), copies, copy_shape, iters, feeder,
                             int(bool(zero_data)), accs, ctypes.byref(t), ctypes.byref(ns), ctypes.byref(mhz)))
    return t.value, ns.value, mhz.value


def wq_calibrate_outliers(x, s=None, rotate: bool = True, transform_order: int = WQ_ORDER_SMOOTH_ROTATE,
                          n_top: int = 0, stream=None):
    """Pooled channel energy z(c) of the transformed calibration activations x (device bf16
    [M, K]) and its Top-K channels: returns device tensors (z fp64 [K], omega int32 [n_top])."""
    import torch
    M, K = x.shape
    dev = x.device
    z = torch.empty(K, dtype=torch.float64, device=dev)
    om = torch.empty(max(n_top, 1), dtype=torch.int32, device=dev)
    s_t = None
    if s is not None:
        s_t = torch.as_tensor(np.asarray(s, np.float32)).to(dev)
    ws = _alloc_workspace(int(lib().wq_calibration_workspace_bytes(M, K)), dev)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else None)
    _check(lib().wq_calibrate_outliers(ptr(x), M, K, ptr(s_t), int(bool(rotate)), int(transform_order), int(n_top),
                                       ptr(z), ptr(om), ptr(ws), ws.numel(), ctypes.c_void_p(_stream_ptr(stream))))
    return z, om[:n_top]


def wq_check_device_error(w: Weights, stream=None):
    _check(lib().wq_check_device_error(ctypes.c_void_p(w.handle), ctypes.c_void_p(_stream_ptr(stream))))


def wq_free_weights(w: Weights):
    if w.handle:
        lib().wq_free_weights(ctypes.c_void_p(w.handle))
        w.handle = None


def mma_scales_to_rowmajor(sf_mma: np.ndarray, M: int, K: int) -> np.ndarray:
    """Decode the documented tcgen05 block-scale layout (wq.h) into [M, K/16]."""
    sf = np.asarray(sf_mma, np.uint8).reshape(-1)
    m = np.arange(M)[:, None]
    b = np.arange(K // 16)[None, :]
    off = ((m // 128) * (K // 64) + b // 4) * 512 + (m % 32) * 16 + ((m % 128) // 32) * 4 + (b % 4)
    return sf[off]


# ------------------------------------------------------------------ selective 8-bit layers
def wq_linear_forward_w8a8(w: Weights, x, y=None, workspace=None, stream=None):
    """y[M, N] bf16 = W8A8 projection of x[M, K] bf16 (handle prepared with WQ_MODE_W8A8)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous() and x.shape[-1] == w.K
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, w.N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _alloc_workspace(wq_workspace_bytes(w, M), x.device)
    _check(lib().wq_linear_forward_w8a8(ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), M,
                                        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                                        workspace.numel(), ctypes.c_void_p(_stream_ptr(stream))))
    return y


def wq_quantize_activations_w8a8(w: Weights, x, stream=None):
    """8-bit quantiser alone: (codes, scale fp32 [M]) on the device; codes are bf16 [M, K] holding
    integers (WQ_MODE_W8A8) or e4m3 bytes uint8 [M, K] (WQ_MODE_W8A8_FP8)."""
    import torch
    M, K = x.shape
    fp8 = w.cfg.mode == WQ_MODE_W8A8_FP8
    codes = torch.empty((M, K), dtype=torch.uint8 if fp8 else torch.bfloat16, device=x.device)
    scale = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(lib().wq_quantize_activations_w8a8(ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), M,
                                              ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scale.data_ptr()),
                                              ctypes.c_void_p(_stream_ptr(stream))))
    return codes, scale


def wq_export_weights_w8a8(w: Weights):
    """(q [N, K], w [N]): int8 values, or e4m3 codes as uint8 for WQ_MODE_W8A8_FP8."""
    q = np.zeros((w.N, w.K), np.uint8 if w.cfg.mode == WQ_MODE_W8A8_FP8 else np.int8)
    sc = np.zeros(w.N, np.float32)
    _check(lib().wq_export_weights_w8a8(ctypes.c_void_p(w.handle), q.ctypes.data_as(ctypes.c_void_p),
                                        sc.ctypes.data_as(ctypes.c_void_p)))
    return q, sc


# ------------------------------------------------------------------ VAE Conv3d
@dataclass
class ConvWeights(Weights):
    C_in: int = 0


def wq_prepare_conv3d(w, pad: int = 1, stream=None) -> ConvWeights:
    """Quantise a [C_out, C_in, kt, kh, kw] fp32 kernel for the implicit-GEMM Conv3d."""
    w = np.ascontiguousarray(w.detach().cpu().numpy() if hasattr(w, "numpy") else w, dtype=np.float32)
    Co, Ci, kt, kh, kw = w.shape
    out = ctypes.c_void_p()
    _check(lib().wq_prepare_conv3d(w.ctypes.data_as(ctypes.c_void_p), Ci, Co, kt, kh, kw, int(pad),
                                   ctypes.c_void_p(_stream_ptr(stream)), ctypes.byref(out)))
    return ConvWeights(out.value, wq_config(kt * kh * kw * Ci, Co, 0, 0, 0, WQ_MODE_W4A4, 0, 0.0, 0), Ci)


def wq_conv3d_workspace_bytes(w: ConvWeights, B: int, D: int, H: int, W: int) -> int:
    return int(lib().wq_conv3d_workspace_bytes(ctypes.c_void_p(w.handle), B, D, H, W))


def wq_conv3d_forward(w: ConvWeights, x, y=None, workspace=None, stream=None):
    """y [B, C_out, D, H, W] bf16 = conv3d(x [B, C_in, D, H, W] bf16), 3x3x3, padding 1."""
    import torch
    B, C, D, H, W = x.shape
    if y is None:
        y = torch.empty((B, w.N, D, H, W), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _alloc_workspace(wq_conv3d_workspace_bytes(w, B, D, H, W), x.device)
    _check(lib().wq_conv3d_forward(ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), B, D, H, W,
                                   ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                                   workspace.numel(), ctypes.c_void_p(_stream_ptr(stream))))
    return y


def wq_quantize_conv3d_input(w: ConvWeights, x, stream=None):
    import torch
    B, C, D, H, W = x.shape
    V = B * D * H * W
    codes = torch.empty((V, C // 2), dtype=torch.uint8, device=x.device)
    scales = torch.empty((V, C // 16), dtype=torch.uint8, device=x.device)
    g = torch.empty(1, dtype=torch.float32, device=x.device)
    ws = _alloc_workspace(wq_conv3d_workspace_bytes(w, B, D, H, W), x.device)
    _check(lib().wq_quantize_conv3d_input(ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), B, D, H, W,
                                          ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scales.data_ptr()),
                                          ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                          ctypes.c_void_p(_stream_ptr(stream))))
    return codes, scales, g
