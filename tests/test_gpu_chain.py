"""GPU parity of the chained projection: the next layer's NVFP4 input produced in this layer's
GEMM epilogue (wq_linear_forward_chain) against the oracle's chain (this layer's output rounded
once to bf16, then the next layer's quantiser with its fixed tensor scale).

Bar: codes, e4m3 scales, tensor scales and fp16 kept channels bit-exact against the oracle on a
first layer whose 4-bit product is exact in fp32 (so both sides round the same output value);
bit-exact against the separate quantiser run on the stored bf16 output for arbitrary layers; the
second layer's y within the usual tolerance.
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


def exact_first_layer(M, K, N, seed):
    """Inputs on which NVFP4 quantisation is lossless and the product exact in fp32: each
    activation row holds 2688 2^E (so its tensor scale is 2^E) and blocks of e2m1 grid values
    times a scale in {1/2, 1, 2, 4}; the weight likewise with one 2688 2^F entry; the bias a
    multiple of 2^(F-2).  Every accumulator sum stays below 2^24 of its smallest unit."""
    rng = np.random.default_rng(seed)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])

    def blocks(rows, n, big_at):
        a = np.zeros((rows, n), np.float64)
        for i in range(rows):
            for b in range(n // 16):
                c = rng.choice(grid, 16) * rng.choice([-1.0, 1.0], 16)
                c[rng.integers(16)] = 6.0 * rng.choice([-1.0, 1.0])
                a[i, 16 * b:16 * b + 16] = c * rng.choice([0.5, 1.0, 2.0, 4.0])
        for (i, j) in big_at:                    # the block of the big entry holds only it
            b = j // 16
            a[i, 16 * b:16 * b + 16] = 0.0
            a[i, j] = 2688.0
        return a
    E = rng.integers(-2, 3, M)
    x = blocks(M, K, [(m, 0) for m in range(M)]) * (2.0 ** E)[:, None]
    F = -6
    Wt = blocks(N, K, [(int(rng.integers(N)), int(rng.integers(K)))]) * 2.0 ** F     # [N, K], per column
    bias = rng.integers(-64, 65, N) * 2.0 ** (F - 2)
    return x.astype(np.float32), np.ascontiguousarray(Wt.T).astype(np.float32), bias.astype(np.float32)


def next_layer(K, N, seed, n_out, rotate_first=False):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    s = np.exp(rng.uniform(-0.7, 0.7, K)).astype(np.float32)
    omega = np.sort(rng.choice(K, n_out, replace=False)).astype(np.int32) if n_out else None
    b = (rng.standard_normal(N) * 0.02).astype(np.float32)
    return W, s, omega, b


def calibrated_g(y, s, rotate, omega, rotate_first):
    """A fixed tensor scale for the next layer: the amax of its transformed input / 2688, from the
    oracle's own output, times 1.25 (headroom, as a calibration from other data would leave)."""
    aq = oracle.chain_quantize(y, s, rotate, omega, 1.0, rotate_first)
    with oracle.transform_order(rotate_first):
        per = oracle.quantize_act(oracle.bf16_bits_from_f64(y), s, rotate, omega, per_tensor=True)
    return float(np.float32(per.g[0] * np.float32(1.25))), aq


@pytest.mark.parametrize("M,rotate_first,n_out", [(200, False, 12), (96, True, 0), (300, False, 41)])
def test_chain_bitexact_against_oracle(M, rotate_first, n_out):
    K, N, N2 = 256, 512, 256
    x, W, bias = exact_first_layer(M, K, N, 5 + M)
    xb = wl.bf16_bits(x)
    assert np.array_equal(wl.bf16_from_bits(xb), x)
    w1 = wq.wq_prepare_weights(K, N, W, bias, rotate=False)
    W2, s2, om2, b2 = next_layer(N, N2, 7 + M, n_out)
    # the oracle's first layer: exact by construction
    L1 = wl.LayerInputs(wl.WORKLOADS["expert"], wl.LayerSpec("l1", K, N), M, xb, W, bias, None, None, None,
                        np.zeros(0, np.int32), False)
    y1, *_ = oracle.reference_forward(L1)
    g2, _ = calibrated_g(y1, s2, True, om2, rotate_first)
    w2 = wq.wq_prepare_weights(N, N2, W2, b2, s2, omega=om2, rotate=True, act_scale=wq.WQ_ACT_SCALE_STATIC,
                               act_gscale=g2, transform_order=int(rotate_first))
    xd = x_dev(xb)
    codes, sf, g, xo = wq.wq_linear_forward_chain(w1, w2, xd)
    y1_gpu = wq.wq_linear_forward(w1, xd)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w1)
    # the first layer's stored output is the oracle's, rounded once (the construction is exact)
    assert np.array_equal(y1_gpu.cpu().view(torch.int16).numpy().view(np.uint16), oracle.bf16_bits_from_f64(y1))
    aq = oracle.chain_quantize(y1, s2, True, om2, g2, rotate_first)
    assert np.all(g.cpu().numpy() == np.float32(g2))
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    assert np.array_equal(wq.mma_scales_to_rowmajor(sf.cpu().numpy(), M, N), aq.scales)
    if n_out:
        xo_np = xo.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(xo_np[:, :n_out], aq.x_omega) and not xo_np[:, n_out:].any()
    # the second layer on the chained input, against the oracle forward with that fixed g
    y2 = wq.wq_linear_forward_quantized(w2, codes, sf, g, None, xo)
    torch.cuda.synchronize()
    with oracle.transform_order(rotate_first):
        wo2 = oracle.prepare_weights(W2, s2, None, None, om2, True)
    y2_ref = oracle.linear_forward(aq, wo2, None, b2, per_tensor_act=True)
    y1_f = wl.bf16_from_bits(oracle.bf16_bits_from_f64(y1)).astype(np.float64)
    tol = 1e-3 * (np.abs(y2_ref) + np.linalg.norm(y1_f, axis=1)[:, None] *
                  np.linalg.norm(W2.astype(np.float64), axis=0)[None, :] / np.sqrt(N)) + 2.0 ** -8 * np.abs(y2_ref)
    err = np.abs(y2.float().cpu().numpy().astype(np.float64) - y2_ref)
    assert (err <= tol).all(), f"{(err > tol).sum()} outside tolerance"


@pytest.mark.parametrize("case", ["dit", "dit_rotate_first"])
def test_chain_matches_the_separate_quantiser(case, tuning):
    """On arbitrary layers (rank, kept channels, smoothing) the epilogue's codes equal those of the
    stand-alone quantiser run on the bf16 output the same GEMM schedule stores."""
    tuning("WQ_GEMM_WIDE", 1)
    L = wl.make_layer_inputs("video_dit", M=300, K=512, N=512, rank=32, n_omega=16)
    w1 = wq.wq_prepare_weights(512, 512, L.W, L.bias, L.s, L.L1, L.L2, L.omega, rotate=True)
    rf = case.endswith("first")
    W2, s2, om2, b2 = next_layer(512, 192, 3, 20)
    w2 = wq.wq_prepare_weights(512, 192, W2, b2, s2, omega=om2, rotate=True, act_scale=wq.WQ_ACT_SCALE_STATIC,
                               act_gscale=0.01, transform_order=int(rf))
    xd = x_dev(L.x_bits)
    codes, sf, g, xo = wq.wq_linear_forward_chain(w1, w2, xd)
    y1 = wq.wq_linear_forward(w1, xd)
    c2, s2q, g2q, xo2, _ = wq.wq_quantize_activations(w2, y1, wq.WQ_SCALE_LAYOUT_MMA)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w1)
    assert torch.equal(codes, c2) and torch.equal(sf, s2q) and torch.equal(g, g2q)
    assert torch.equal(xo, xo2)


def test_chain_rejects_unsupported_next_layers():
    W = np.zeros((256, 256), np.float32)
    w1 = wq.wq_prepare_weights(256, 256, W, rotate=False)
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    w_row = wq.wq_prepare_weights(256, 128, np.zeros((256, 128), np.float32), rotate=True)
    with pytest.raises(wq.WqError) as e:
        wq.wq_linear_forward_chain(w1, w_row, x)
    assert e.value.status == wq.WQ_ERR_UNSUPPORTED
    L1 = np.ones((256, 16), np.float32)
    L2 = np.ones((16, 128), np.float32)
    w_rank = wq.wq_prepare_weights(256, 128, np.zeros((256, 128), np.float32), L1=L1, L2=L2, rotate=True,
                                   act_scale=wq.WQ_ACT_SCALE_STATIC, act_gscale=1.0)
    with pytest.raises(wq.WqError) as e:
        wq.wq_linear_forward_chain(w1, w_rank, x)
    assert e.value.status == wq.WQ_ERR_UNSUPPORTED
    w_bad = wq.wq_prepare_weights(128, 128, np.zeros((128, 128), np.float32), rotate=True,
                                  act_scale=wq.WQ_ACT_SCALE_STATIC, act_gscale=1.0)
    with pytest.raises(wq.WqError):
        wq.wq_linear_forward_chain(w1, w_bad, x)
