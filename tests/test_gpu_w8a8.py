"""GPU parity of the selective 8-bit path (W8A8) against the oracle.

Bar: activation and weight int8 codes and their fp32 scales bit-exact; y within
1e-3 (|y| + ||x_row|| ||w_col|| / sqrt(K)) + 2^-8 |y| (fp32 accumulation of exact products
vs exact int64, plus the bf16 output rounding).
"""
import numpy as np
import pytest
import torch

import oracle
import w4a4_nvfp4_quantized_wq_b300 as wq
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a4_nvfp4_quantized_wq_b300 import build
    build.build_library()
    torch.cuda.set_device(0)


def x_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def prep8(L):
    return wq.wq_prepare_weights(L.spec.K, L.spec.N, L.W, L.bias, L.s, rotate=L.rotate, mode=wq.WQ_MODE_W8A8)


def check_y(L, y, y_ref, rows=None):
    x = L.x_f32 if rows is None else L.x_f32[rows]
    xn = np.linalg.norm(x.astype(np.float64), axis=1)[:, None]
    wn = np.linalg.norm(L.W.astype(np.float64), axis=0)[None, :]
    tol = 1e-3 * (np.abs(y_ref) + xn * wn / np.sqrt(L.spec.K)) + 2.0 ** -8 * np.abs(y_ref)
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - y_ref)
    assert (err <= tol).all(), f"{(err > tol).sum()} outside tolerance, worst excess {np.max(err - tol):.3g}"


CASES8 = {
    "oproj_small": dict(layer=1, M=129, K=2048, N=256),
    "down_small": dict(layer=3, M=40, K=1024, N=160),
    "no_rotate": dict(layer=1, M=64, K=512, N=128, rotate=False),
    "no_smooth": dict(layer=1, M=33, K=640, N=96, smooth=False),
    "m1_k64_n16": dict(layer=1, M=1, K=64, N=16),
}


@pytest.mark.parametrize("case", list(CASES8))
def test_w8a8_codes_scales_and_output(case):
    L = wl.make_layer_inputs("backbone", **CASES8[case])
    w = prep8(L)
    q, sc = wq.wq_export_weights_w8a8(w)
    o8 = oracle.prepare_weights_int8(L.W, L.s, L.rotate)
    assert np.array_equal(q, o8.q) and np.array_equal(sc, o8.scale)
    x = x_dev(L.x_bits)
    codes, a = wq.wq_quantize_activations_w8a8(w, x)
    y = wq.wq_linear_forward_w8a8(w, x)
    wq.wq_check_device_error(w)
    y_ref, aq, _ = oracle.reference_forward_w8a8(L)
    assert np.array_equal(codes.float().cpu().numpy().astype(np.int8), aq.q)
    assert np.array_equal(a.cpu().numpy(), aq.scale)
    check_y(L, y, y_ref)


@pytest.mark.parametrize("split", [1, 2, 8])
@pytest.mark.parametrize("push", ["1", "0"])
def test_w8a8_split_k_schedules(split, push, tuning):
    tuning("WQ_GEMM_SPLIT", str(split))
    tuning("WQ_GEMM_PUSH", push)
    L = wl.make_layer_inputs("backbone", **CASES8["oproj_small"])
    w = prep8(L)
    y = wq.wq_linear_forward_w8a8(w, x_dev(L.x_bits))
    y_ref, *_ = oracle.reference_forward_w8a8(L)
    check_y(L, y, y_ref)


@pytest.mark.parametrize("case", list(CASES8))
def test_w8a8_pair_schedule(case, tuning):
    """The 8-bit layers on the CTA-pair schedule (256 x 256 tiles, kind::f16 pair MMAs)."""
    tuning("WQ_GEMM_WIDE", "1")
    L = wl.make_layer_inputs("backbone", **CASES8[case])
    w = prep8(L)
    y = wq.wq_linear_forward_w8a8(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    y_ref, *_ = oracle.reference_forward_w8a8(L)
    check_y(L, y, y_ref)


@pytest.mark.parametrize("layer_idx", [1, 3])
def test_w8a8_full_size_sampled_rows(layer_idx):
    L = wl.make_layer_inputs("backbone", layer=layer_idx)
    w = prep8(L)
    x = x_dev(L.x_bits)
    y = wq.wq_linear_forward_w8a8(w, x)
    codes, a = wq.wq_quantize_activations_w8a8(w, x)
    wq.wq_check_device_error(w)
    rows = np.sort(np.random.default_rng(200 + layer_idx).choice(L.M, size=24, replace=False))
    y_ref, aq, _ = oracle.reference_forward_w8a8(L, rows=rows)
    assert np.array_equal(codes.float().cpu().numpy()[rows].astype(np.int8), aq.q)
    assert np.array_equal(a.cpu().numpy()[rows], aq.scale)
    check_y(L, y[torch.from_numpy(rows).cuda()], y_ref, rows)
