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


# ------------------------------------------------------------------ FP8 W8A8 (upgraded layers)
def prep_fp8(L):
    return wq.wq_prepare_weights(L.spec.K, L.spec.N, L.W, L.bias, L.s, rotate=L.rotate, mode=wq.WQ_MODE_W8A8_FP8)


# K % 128 == 64 included: the last 128-byte stage is half filled (zeros past K)
CASES_F8 = dict(CASES8, k_tail=dict(layer=1, M=70, K=576, N=144))


@pytest.mark.parametrize("case", list(CASES_F8))
@pytest.mark.parametrize("wide", ["0", "1"])
def test_fp8_w8a8_codes_scales_and_output(case, wide, tuning):
    """QuantWAMs sec. 4.2: FP8 W8A8 for the upgraded layers.  e4m3 weight and activation codes
    and their scales bit-exact against the oracle; y within tolerance, on the single-CTA and the
    CTA-pair GEMM (kind::f8f6f4)."""
    tuning("WQ_GEMM_WIDE", wide)
    L = wl.make_layer_inputs("backbone", **CASES_F8[case])
    w = prep_fp8(L)
    assert (wq.wq_gemm_schedule(w, L.M) == wq.WQ_GEMM_WIDE) == (wide == "1")
    q, sc = wq.wq_export_weights_w8a8(w)
    of = oracle.prepare_weights_fp8(L.W, L.s, L.rotate)
    assert np.array_equal(q, of.q) and np.array_equal(sc, of.scale)
    x = x_dev(L.x_bits)
    codes, a = wq.wq_quantize_activations_w8a8(w, x)
    y = wq.wq_linear_forward_w8a8(w, x)
    wq.wq_check_device_error(w)
    y_ref, aq, _ = oracle.reference_forward_fp8(L)
    assert np.array_equal(codes.cpu().numpy(), aq.q)
    assert np.array_equal(a.cpu().numpy(), aq.scale)
    check_y(L, y, y_ref)


@pytest.mark.parametrize("split", [2, 8])
def test_fp8_w8a8_split_k(split, tuning):
    tuning("WQ_GEMM_SPLIT", str(split))
    L = wl.make_layer_inputs("backbone", **CASES8["down_small"])
    w = prep_fp8(L)
    y = wq.wq_linear_forward_w8a8(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    y_ref, *_ = oracle.reference_forward_fp8(L)
    check_y(L, y, y_ref)


def test_fp8_w8a8_ties_and_saturation():
    """Quotients exactly on e4m3 midpoints (s = 1, no rotation; a row maximum of 448 gives a = 1):
    round to even, and the row maximum itself lands on 448."""
    K = 256
    mids = []
    for e in range(1, 14):
        for m in range(7):
            lo = (1 + m / 8) * 2.0 ** (e - 7)
            mids.append(lo + 2.0 ** (e - 7) / 16)
    x = np.zeros((4, K), np.float32)
    for r in range(4):
        x[r, 0] = 448.0
        vals = np.array(mids[r * 60:(r + 1) * 60], np.float32)
        x[r, 1:1 + vals.size] = vals * np.where(np.arange(vals.size) % 2, -1, 1)
    bits = wl.bf16_bits(x)
    W = np.random.default_rng(2).standard_normal((K, 32)).astype(np.float32) * 0.02
    w = wq.wq_prepare_weights(K, 32, W, rotate=False, mode=wq.WQ_MODE_W8A8_FP8)
    codes, a = wq.wq_quantize_activations_w8a8(w, x_dev(bits))
    torch.cuda.synchronize()
    aq = oracle.quantize_act_fp8(bits, None, False)
    assert np.all(aq.scale == 1.0)
    assert np.array_equal(codes.cpu().numpy(), aq.q)
    assert np.array_equal(a.cpu().numpy(), aq.scale)


def test_fp8_w8a8_full_size_down_projection():
    """The language backbone's down projection (K = 16384) in FP8: every row's codes bit-exact,
    y on one row per 128-row tile."""
    L = wl.make_layer_inputs("backbone", layer=3)
    w = prep_fp8(L)
    x = x_dev(L.x_bits)
    y = wq.wq_linear_forward_w8a8(w, x)
    codes, a = wq.wq_quantize_activations_w8a8(w, x)
    wq.wq_check_device_error(w)
    aq = oracle.quantize_act_fp8(L.x_bits, L.s, L.rotate)
    assert np.array_equal(codes.cpu().numpy(), aq.q) and np.array_equal(a.cpu().numpy(), aq.scale)
    rows = np.array(sorted({0, L.M - 1} | {t + 7 for t in range(0, L.M, 128)}))
    y_ref, *_ = oracle.reference_forward_fp8(L, rows=rows)
    check_y(L, y[torch.from_numpy(rows).cuda()], y_ref, rows)
