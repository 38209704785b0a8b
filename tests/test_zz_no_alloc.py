"""The no-allocation forward (wq_linear_forward_noalloc) against the ordinary forward.

Callers such as engine plugins or real-time control loops cannot allocate device memory
after start-up, so this entry point takes its scratch from a static device array inside
the library.  The test calls it through the C ABI twice in a row -- with different
layers, so stale scratch from the first call would show -- and compares each output with
wq_linear_forward on the same inputs under the parity tolerance used for the forward.
"""
import ctypes

import numpy as np
import pytest
import torch

import w4a4_nvfp4_quantized_wq_b300 as wq
import workloads as wl

pytestmark = pytest.mark.gpu


def _y_tolerance(L, y_ref):
    xn = np.linalg.norm(L.x_f32.astype(np.float64), axis=1)[:, None]
    wn = np.linalg.norm(L.W.astype(np.float64), axis=0)[None, :]
    return 1e-3 * (np.abs(y_ref) + xn * wn / np.sqrt(L.spec.K)) + 2.0 ** -8 * np.abs(y_ref)


def test_noalloc_forward_matches_forward_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a4_nvfp4_quantized_wq_b300 import build
    build.build_library()
    torch.cuda.set_device(0)
    L = wq.lib()
    cases = [wl.make_layer_inputs("expert", layer=1),                                   # K=4096 -> 1024
             wl.make_layer_inputs("video_dit", M=300, K=512, N=272, rank=32, n_omega=64)]
    for Li in cases:
        w = wq.wq_prepare_weights(Li.spec.K, Li.spec.N, Li.W, Li.bias, Li.s, Li.L1, Li.L2,
                                  Li.omega if Li.omega.size else None, rotate=Li.rotate)
        x = torch.from_numpy(Li.x_bits.view(np.int16)).view(torch.bfloat16).cuda()
        y_ref = wq.wq_linear_forward(w, x)
        y = torch.full((Li.M, Li.spec.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = L.wq_linear_forward_noalloc(ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), Li.M,
                                         ctypes.c_void_p(y.data_ptr()),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == wq.WQ_OK, wq.wq_last_error()
        torch.cuda.synchronize()
        wq.wq_check_device_error(w)
        a = y.float().cpu().numpy().astype(np.float64)
        b = y_ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a))
        assert np.all(np.abs(a - b) <= _y_tolerance(Li, b))
    # a size beyond the static array is refused with a clear error
    big = 1 << 20
    rc = L.wq_linear_forward_noalloc(ctypes.c_void_p(w.handle), ctypes.c_void_p(x.data_ptr()), big,
                                     ctypes.c_void_p(y.data_ptr()), None)
    assert rc == wq.WQ_ERR_UNSUPPORTED and "scratch" in wq.wq_last_error()
