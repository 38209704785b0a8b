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


def _cfg(K=256, N=128, r=0, no=0, rot=1, mode=0, act=0, g=0.0, order=0, proj=0):
    return wq.wq_config(K, N, r, no, rot, mode, act, g, order, proj)


@pytest.mark.parametrize("cfg,status", [
    (dict(K=100), wq.WQ_ERR_UNSUPPORTED),
    (dict(K=32768), wq.WQ_ERR_UNSUPPORTED),
    (dict(N=24), wq.WQ_ERR_UNSUPPORTED),
    (dict(r=65), wq.WQ_ERR_UNSUPPORTED),
    (dict(no=65), wq.WQ_ERR_UNSUPPORTED),
    (dict(K=64, no=64, r=0), None),                      # accepted shape (checked below to succeed)
    (dict(mode=1, r=16), wq.WQ_ERR_UNSUPPORTED),
    (dict(mode=1, act=1), wq.WQ_ERR_UNSUPPORTED),
    (dict(mode=4), wq.WQ_ERR_INVALID),
    (dict(mode=3, act=1), wq.WQ_ERR_UNSUPPORTED),
    (dict(mode=2, r=16), wq.WQ_ERR_UNSUPPORTED),
    (dict(mode=2, order=1), wq.WQ_ERR_UNSUPPORTED),
    (dict(rot=2), wq.WQ_ERR_INVALID),
    (dict(K=-64), wq.WQ_ERR_INVALID),
    (dict(act=3), wq.WQ_ERR_INVALID),
    (dict(act=2, g=0.0), wq.WQ_ERR_INVALID),
    (dict(act=2, g=float("inf")), wq.WQ_ERR_INVALID),
    (dict(order=2), wq.WQ_ERR_INVALID),
    (dict(mode=1, order=1), wq.WQ_ERR_UNSUPPORTED),
    (dict(proj=2, r=16), wq.WQ_ERR_INVALID),
    (dict(proj=1), wq.WQ_ERR_UNSUPPORTED),                # no branch to project on
    (dict(proj=1, r=16, act=1), wq.WQ_ERR_UNSUPPORTED),
    (dict(proj=1, r=16, order=1), wq.WQ_ERR_UNSUPPORTED),
    (dict(proj=1, r=16, mode=3), wq.WQ_ERR_UNSUPPORTED),
])
def test_prepare_rejects_bad_config(cfg, status):
    if status is None:
        pytest.skip("accepted configuration: preparing it needs a device")
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
                 "WQ_GEMM_WIDE_DB",
                 "WQ_QUANT_CLUSTER", "WQ_QUANT_STREAM", "WQ_QUANT_RESIDENT"):
        assert int(defs[name]) == getattr(wq, name), name


def test_tuning_knobs_through_the_abi():
    """Schedule knobs: the environment is read once, then wq_set_tuning alone changes them."""
    L = wq.lib()
    old = L.wq_get_tuning(b"WQ_QUANT_SPLIT")
    assert L.wq_set_tuning(b"WQ_QUANT_SPLIT", 4) == wq.WQ_OK
    assert L.wq_get_tuning(b"WQ_QUANT_SPLIT") == 4
    os.environ["WQ_QUANT_SPLIT"] = "8"              # no longer read
    try:
        assert L.wq_get_tuning(b"WQ_QUANT_SPLIT") == 4
    finally:
        del os.environ["WQ_QUANT_SPLIT"]
    assert L.wq_set_tuning(b"WQ_QUANT_SPLIT", old) == wq.WQ_OK
    old_db = L.wq_get_tuning(b"WQ_GEMM_DB")
    if "WQ_GEMM_DB" not in os.environ:
        assert old_db == -1                          # automatic unless the environment pins it
    assert L.wq_set_tuning(b"WQ_GEMM_DB", 0) == wq.WQ_OK and L.wq_get_tuning(b"WQ_GEMM_DB") == 0
    assert L.wq_set_tuning(b"WQ_GEMM_DB", old_db) == wq.WQ_OK
    assert L.wq_set_tuning(b"WQ_NOT_A_KNOB", 1) == wq.WQ_ERR_INVALID
    assert "unknown" in wq.wq_last_error()
    assert L.wq_get_tuning(b"WQ_NOT_A_KNOB") == wq.WQ_ERR_INVALID
    assert L.wq_set_tuning(None, 1) == wq.WQ_ERR_INVALID


def test_new_entry_points_reject_bad_arguments_before_device_work():
    L = wq.lib()
    u, x = ctypes.c_int(7), ctypes.c_int(7)
    assert L.wq_side_strides(None, ctypes.byref(u), ctypes.byref(x)) == wq.WQ_ERR_INVALID
    assert L.wq_conv3d_workspace_bytes(None, 1, 8, 8, 8) == 0
    d = ctypes.c_double()
    for args in [(3, 256, 0, 0, 0, 16, 0, 0, 1), (0, 100, 0, 0, 0, 16, 0, 0, 1), (0, 256, 0, 4, 0, 16, 0, 0, 1),
                 (0, 256, 0, 0, 2, 16, 0, 0, 1), (0, 256, 0, 0, 0, 0, 0, 0, 1), (0, 256, 0, 1, 0, 16, 3, 0, 1),
                 (0, 256, 0, 1, 1, 16, 2, 0, 1), (0, 256, 0, 0, 0, 16, 0, 0, 2), (0, 128, 0, 0, 0, 16, 0, 0, 3)]:
        assert L.wq_mma_peak(*args, ctypes.byref(d), ctypes.byref(d), ctypes.byref(d)) == wq.WQ_ERR_INVALID
    w = np.zeros((16, 128, 3, 3, 3), np.float32)
    out = ctypes.c_void_p()
    vp = w.ctypes.data_as(ctypes.c_void_p)
    assert L.wq_prepare_conv3d(vp, 128, 16, 1, 3, 3, 1, None, ctypes.byref(out)) == wq.WQ_ERR_UNSUPPORTED
    assert L.wq_prepare_conv3d(vp, 128, 16, 3, 3, 3, 0, None, ctypes.byref(out)) == wq.WQ_ERR_UNSUPPORTED
    assert L.wq_prepare_conv3d(vp, 128, 16, 3, 3, 3, -1, None, ctypes.byref(out)) == wq.WQ_ERR_INVALID
    assert out.value is None


def test_side_width_rule_in_the_binding_docs():
    """The stored widths of U and x_Omega: counts rounded up to 16, 32 or 64."""
    txt = open(os.path.join(ROOT, "include", "wq.h")).read()
    assert "rounded up to 16, 32 or 64" in txt
