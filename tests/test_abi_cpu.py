"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
and rejects invalid arguments with status codes before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import w4a4_nvfp4_quantized_wq_b300 as wq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from w4a4_nvfp4_quantized_wq_b300 import build
    build.build_library()


def _declared():
    txt = open(os.path.join(ROOT, "include", "wq.h")).read()
    return re.findall(r"WQ_API\s+[\w\s\*]+?\b(wq_\w+)\s*\(", txt)


def test_header_declarations_match_binding():
    assert sorted(_declared()) == sorted(wq.EXPORTED)


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(wq.LIB_PATH)
    for name in _declared():
        assert hasattr(L, name), name


def _cfg(K=256, N=128, r=0, no=0, rot=1, mode=0):
    return wq.wq_config(K, N, r, no, rot, mode)


@pytest.mark.parametrize("cfg,status", [
    (dict(K=100), wq.WQ_ERR_UNSUPPORTED),
    (dict(K=32768), wq.WQ_ERR_UNSUPPORTED),
    (dict(N=24), wq.WQ_ERR_UNSUPPORTED),
    (dict(r=8), wq.WQ_ERR_UNSUPPORTED),
    (dict(no=20), wq.WQ_ERR_UNSUPPORTED),
    (dict(mode=1, r=16), wq.WQ_ERR_UNSUPPORTED),
    (dict(mode=2), wq.WQ_ERR_INVALID),
    (dict(rot=2), wq.WQ_ERR_INVALID),
    (dict(K=-64), wq.WQ_ERR_INVALID),
])
def test_prepare_rejects_bad_config(cfg, status):
    c = _cfg(**cfg)
    W = np.zeros((max(c.K, 1), max(c.N, 1)), np.float32)
    out = ctypes.c_void_p()
    rc = wq.lib().wq_prepare_weights(ctypes.byref(c), W.ctypes.data_as(ctypes.c_void_p), None, None, None, None,
                                     None, None, ctypes.byref(out))
    assert rc == status, wq.wq_last_error()
    assert out.value is None
    assert wq.wq_last_error()


def test_prepare_rejects_null_and_unsorted_inputs():
    c = _cfg(no=16)
    W = np.zeros((256, 128), np.float32)
    out = ctypes.c_void_p()
    L = wq.lib()
    assert L.wq_prepare_weights(ctypes.byref(c), None, None, None, None, None, None, None,
                                ctypes.byref(out)) == wq.WQ_ERR_INVALID
    om = np.arange(16, dtype=np.int32)[::-1].copy()
    assert L.wq_prepare_weights(ctypes.byref(c), W.ctypes.data_as(ctypes.c_void_p), None, None, None, None,
                                om.ctypes.data_as(ctypes.c_void_p), None, ctypes.byref(out)) == wq.WQ_ERR_INVALID
    om = np.arange(16, dtype=np.int32) + 250
    assert L.wq_prepare_weights(ctypes.byref(c), W.ctypes.data_as(ctypes.c_void_p), None, None, None, None,
                                om.ctypes.data_as(ctypes.c_void_p), None, ctypes.byref(out)) == wq.WQ_ERR_INVALID
    s = -np.ones(256, np.float32)
    c0 = _cfg()
    assert L.wq_prepare_weights(ctypes.byref(c0), W.ctypes.data_as(ctypes.c_void_p), None,
                                s.ctypes.data_as(ctypes.c_void_p), None, None, None, None,
                                ctypes.byref(out)) == wq.WQ_ERR_INVALID
    c1 = _cfg(r=16)
    assert L.wq_prepare_weights(ctypes.byref(c1), W.ctypes.data_as(ctypes.c_void_p), None, None, None, None,
                                None, None, ctypes.byref(out)) == wq.WQ_ERR_INVALID


def test_null_handle_calls_fail_cleanly():
    L = wq.lib()
    assert L.wq_workspace_bytes(None, 16) == 0
    assert L.wq_linear_forward(None, None, 4, None, None, 0, None) == wq.WQ_ERR_INVALID
    assert L.wq_quantize_activations(None, None, 4, 0, None, None, None, None, None, None) == wq.WQ_ERR_INVALID
    assert L.wq_export_weights(None, None, None, None, None, None, None) == wq.WQ_ERR_INVALID
    L.wq_free_weights(None)


def test_path_queries_and_self_test_reject_bad_arguments():
    """The host queries of the path a forward takes, and the wait self-test's output checks,
    fail with status codes (and a message) before any device work."""
    L = wq.lib()
    for fn in (L.wq_forward_path, L.wq_gemm_schedule, L.wq_quant_schedule):
        assert fn(None, 16) == wq.WQ_ERR_INVALID
        assert wq.wq_last_error()
    assert L.wq_selftest_wait_timeout(None, None, None) == wq.WQ_ERR_INVALID
    assert "NULL" in wq.wq_last_error()


def test_path_constants_match_the_header():
    txt = open(os.path.join(ROOT, "include", "wq.h")).read()
    defs = dict(re.findall(r"#define\s+(WQ_\w+)\s+(-?\d+)", txt))
    for name in ("WQ_PATH_TWO_KERNEL", "WQ_PATH_FUSED", "WQ_GEMM_SINGLE", "WQ_GEMM_SPLITK", "WQ_GEMM_WIDE",
                 "WQ_QUANT_CLUSTER", "WQ_QUANT_STREAM"):
        assert int(defs[name]) == getattr(wq, name), name
