"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against mathematics the pages (or the NVFP4
format definition they name) fix: a dense matrix definition, a closed form, an
invariant, an exhaustive independent restatement, or a library routine.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

import oracle
import workloads as wlmod

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden_formats():
    tab = {"e2m1": {}, "e4m3": {}}
    with open(os.path.join(HERE, "golden", "nvfp4_formats.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, code, val = line.split()
            tab[fmt][int(code)] = float(val)
    return tab


GOLD = _golden_formats()


# ------------------------------------------------------------------ FWHT
# FoldQuantVLA, Key Contribution 2: block Hadamard rotation applied via the FWHT, beta = 64.
def test_fwht_equals_dense_sylvester_matrix():
    H = hadamard(64).astype(np.float64) / 8.0
    rng = np.random.default_rng(11)
    for _ in range(20):
        v = rng.standard_normal(64).astype(np.float32)
        got = oracle.fwht64_f32(v).astype(np.float64)
        ref = H @ v.astype(np.float64)
        assert np.max(np.abs(got - ref)) <= 1e-6 * np.max(np.abs(ref))
        got64 = oracle.fwht64_f64(v.astype(np.float64))
        assert np.max(np.abs(got64 - ref)) <= 1e-13 * np.max(np.abs(ref))


def test_fwht_basis_vectors_give_hadamard_rows_exactly():
    H = hadamard(64).astype(np.float32) / np.float32(8.0)
    for i in range(64):
        e = np.zeros(64, np.float32)
        e[i] = 1.0
        assert np.array_equal(oracle.fwht64_f32(e), H[:, i])


def test_fwht_self_inverse_and_orthonormal():
    rng = np.random.default_rng(12)
    for _ in range(50):
        v = (rng.standard_normal(64) * 10 ** rng.uniform(-3, 3)).astype(np.float32)
        w = oracle.fwht64_f32(v)
        np.testing.assert_allclose(np.linalg.norm(w.astype(np.float64)),
                                   np.linalg.norm(v.astype(np.float64)), rtol=1e-6)
        back = oracle.fwht64_f32(w)
        ulp = np.spacing(np.max(np.abs(v)))
        assert np.max(np.abs(back - v)) <= 4 * ulp


# ------------------------------------------------------------------ formats
def test_e2m1_grid_literal():
    for code, val in GOLD["e2m1"].items():
        d = oracle.e2m1_decode(code)
        assert d == val and np.signbit(d) == np.signbit(val), (code, d, val)
        assert oracle.e2m1_encode(val) == code


def test_e4m3_points_literal():
    for code, val in GOLD["e4m3"].items():
        assert oracle.e4m3_decode(code) == val
        assert oracle.e4m3_encode(val) == code


def test_e2m1_ties_round_to_even_code():
    # midpoints of the grid -> the neighbour with the even magnitude code
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 6.0: 7, 7.0: 7, 1e30: 7,
             -0.1: 8, -0.25: 8, -0.75: 10, -5.0: 14, -100.0: 15}
    for v, c in cases.items():
        assert oracle.e2m1_encode(v) == c, (v, oracle.e2m1_encode(v), c)


@pytest.fixture(scope="module")
def pinlib():
    src = os.path.join(HERE, "pins", "rounding_pin.c")
    out = os.path.join(HERE, "pins", "librounding_pin.so")
    if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               src, "-o", out, "-lm"])
    L = ctypes.CDLL(out)
    L.pin_e2m1_all.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    L.pin_e2m1_all.restype = ctypes.c_long
    L.pin_e4m3_all.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    L.pin_e4m3_all.restype = ctypes.c_long
    return L


def test_e2m1_encoder_exhaustive_against_ieee_rounding(pinlib):
    first = ctypes.c_uint32(0)
    fn = ctypes.cast(oracle.lib().orc_e2m1_encode, ctypes.c_void_p)
    bad = pinlib.pin_e2m1_all(fn, ctypes.byref(first))
    assert bad == 0, f"{bad} mismatches, first fp32 bits {first.value:#010x}"


def test_e4m3_encoder_exhaustive_against_ieee_rounding(pinlib):
    first = ctypes.c_uint32(0)
    fn = ctypes.cast(oracle.lib().orc_e4m3_encode, ctypes.c_void_p)
    bad = pinlib.pin_e4m3_all(fn, ctypes.byref(first))
    assert bad == 0, f"{bad} mismatches, first fp32 bits {first.value:#010x}"


def test_e4m3_encoder_matches_torch_float8_in_range():
    # torch's fp32 -> float8_e4m3fn is round-to-nearest-even; compare where it is finite
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.uniform(0, 448, 200000), 2.0 ** rng.uniform(-12, 8.8, 200000)]).astype(np.float32)
    v = v[v <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(a)) for a in v[:40000]], np.uint8)
    assert np.array_equal(got, ref[:40000])


def test_bf16_from_f64_matches_torch_on_fp32_values():
    rng = np.random.default_rng(6)
    v = (rng.standard_normal(20000) * 10 ** rng.uniform(-30, 30, 20000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.uint16).numpy()
    L = oracle.lib()
    got = np.array([L.orc_bf16_from_f64(float(a)) for a in v], np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ the quantiser
def _dec_table():
    e2 = np.array([GOLD["e2m1"][c] for c in range(16)], np.float64)
    return e2


def _dequant(codes, scales, K):
    """Test-side dequantisation from the golden grid (independent of the oracle)."""
    e2 = _dec_table()
    lo = codes & 15
    hi = codes >> 4
    el = np.empty(codes.shape[:-1] + (K,), np.float64)
    el[..., 0::2] = e2[lo]
    el[..., 1::2] = e2[hi]
    sc = np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)
    return el * np.repeat(sc[scales], 16, axis=-1)


def test_representable_blocks_round_trip_exactly():
    """A block built from representable code x scale values (with g = 1) quantises
    back to exactly those codes and that scale."""
    rng = np.random.default_rng(7)
    e2 = _dec_table()
    for sc in [1, 8, 9, 40, 56, 57, 90, 119, 125]:
        dsc = oracle.e4m3_decode(sc)
        for _ in range(20):
            codes = rng.integers(0, 16, 16)
            codes[rng.integers(0, 16)] = 7 | (8 * rng.integers(0, 2))   # block max = 6 * scale
            v = (e2[codes] * dsc).astype(np.float32)
            c, s = oracle.nvfp4_quantize(v, 1.0)
            assert s[0] == sc
            got = np.empty(16, np.int64)
            got[0::2] = c & 15
            got[1::2] = c >> 4
            want = codes.copy()
            want[(e2[codes] == 0)] = want[(e2[codes] == 0)] & 8       # +-0 keep their sign
            assert np.array_equal(got, want), (sc, got, want)


def test_constant_row_closed_form():
    """A row of equal values c: after the block FWHT only element 0 of each 64-block
    is non-zero (= 8c); it takes the largest code and scale, all others are zero."""
    for c in [0.5, 1.0, -3.0, 1.5]:
        K = 256
        x = np.full((1, K), c, np.float32)
        aq = oracle.quantize_act(wlmod.bf16_bits(x), None, True)
        deq = _dequant(aq.codes, aq.scales, K)[0]
        # element 0 of each block: code +-6 with scale 448 (largest e4m3)
        assert np.array_equal(deq[0::64], np.full(K // 64, np.copysign(6.0 * 448.0, c)))
        assert not np.delete(deq, np.arange(0, K, 64)).any()
        # g = fp32(8|c| / 2688), so the dequantised value is 8c to within one fp32 rounding
        val = deq[0] * np.float64(aq.g[0])
        assert abs(val - 8 * c) <= 2.0 ** -24 * 8 * abs(c)


def test_zero_row_gives_zero_scale_and_codes():
    x = np.zeros((2, 128), np.uint16)
    aq = oracle.quantize_act(x, None, True)
    assert aq.g.tolist() == [0.0, 0.0]
    assert not aq.codes.any() and not aq.scales.any()


def test_quantiser_brute_force_tiny():
    """Brute force on one 16-block: every code is the nearest point of the scaled grid
    (tie -> even code), and the scale is the nearest e4m3 to bmax/6/g."""
    rng = np.random.default_rng(8)
    e2 = _dec_table()[:8]
    for _ in range(300):
        v = (rng.standard_normal(16) * 10 ** rng.uniform(-2, 2)).astype(np.float32)
        g = np.float32(10 ** rng.uniform(-3, 0))
        c, s = oracle.nvfp4_quantize(v, g)
        t = np.float32(np.float32(np.max(np.abs(v))) / np.float32(6.0)) / g
        sv = np.array([oracle.e4m3_decode(k) for k in range(127)])
        dist = np.abs(sv - np.float64(np.float32(t)))
        best = np.flatnonzero(dist == dist.min())
        exp_sc = 126 if t >= 448 else (best[0] if len(best) == 1 else best[best % 2 == 0][0])
        assert s[0] == exp_sc
        d = np.float32(np.float32(sv[exp_sc]) * g)
        for i in range(16):
            code = (c[i // 2] >> (4 * (i % 2))) & 15
            if d == 0:
                assert code == 0
                continue
            q = np.float64(np.float32(v[i] / d))
            a = min(abs(q), 6.0)
            dd = np.abs(e2 - a)
            cand = np.flatnonzero(dd == dd.min())
            mag = cand[0] if len(cand) == 1 else cand[cand % 2 == 0][0]
            assert code == (mag | (8 if np.signbit(q) else 0)), (v[i], d, code, mag)


# ------------------------------------------------------------------ Proposition 1
@pytest.mark.parametrize("r,n_om", [(0, 0), (16, 0), (0, 16), (16, 16)])
def test_folding_invariance_prop1(r, n_om):
    """FoldQuantVLA Proposition 1: with quantisation disabled, the folded graph
    (x diag(s)^-1 H)(H^T diag(s) W) (+ low-rank + outlier branches) computes x W + b."""
    L = wlmod.make_layer_inputs("tiny", M=8, K=256, N=96, rank=r, n_omega=n_om)
    wq = oracle.prepare_weights(L.W, L.s, L.L1, L.L2, L.omega, True)
    y = oracle.forward_noquant(L.x_bits, L.s, True, L.omega, wq, L.bias)
    ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64)
    if L.bias is not None:
        ref += L.bias
    rel = np.max(np.abs(y - ref)) / np.max(np.abs(ref))
    assert rel <= 1e-5, rel


def test_folding_invariance_detects_unfolded_rotation():
    """Sanity of the pin itself: rotating only one side breaks the identity."""
    L = wlmod.make_layer_inputs("tiny", M=8, K=256, N=96, rank=0, n_omega=0)
    wq = oracle.prepare_weights(L.W, L.s, None, None, None, False)       # weight not rotated
    y = oracle.forward_noquant(L.x_bits, L.s, True, None, wq, None)      # activation rotated
    ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64)
    assert np.max(np.abs(y - ref)) / np.max(np.abs(ref)) > 1e-2


# ------------------------------------------------------------------ reduction to a matmul
def test_plain_case_reduces_to_dequantised_matmul():
    """s = 1, no rotation, r = 0, Omega empty: the oracle forward equals
    (deq(A) gA) @ (deq(W) gW)^T + b computed by numpy from the codes."""
    L = wlmod.make_layer_inputs("expert", M=12, K=256, N=80, rank=0, n_omega=0, smooth=False,
                                rotate=False)
    y, aq, wq, _ = oracle.reference_forward(L)
    A = _dequant(aq.codes, aq.scales, 256) * aq.g.astype(np.float64)[:, None]
    B = _dequant(wq.codes, wq.scales, 256) * np.float64(wq.gW)
    ref = A @ B.T + L.bias.astype(np.float64)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.max(np.abs(ref)))


def test_lowrank_and_outlier_terms_enter_with_the_right_sign():
    """y(with branches) - y(main only) equals U Q + x_Omega W_Omega computed by numpy."""
    L = wlmod.make_layer_inputs("video_dit", M=16, K=256, N=64, rank=16, n_omega=16)
    y, aq, wq, U = oracle.reference_forward(L)
    y0 = oracle.linear_forward(aq, oracle.WeightQuant(wq.codes, wq.scales, wq.gW,
                                                      np.zeros((0, 64), np.uint16),
                                                      np.zeros((256, 0), np.uint16),
                                                      np.zeros((0, 64), np.uint16), wq.Rp,
                                                      wq.W_omega_f32[:0]),
                               None, None)
    side = (wlmod.bf16_from_bits(U).astype(np.float64) @ wlmod.bf16_from_bits(wq.Q).astype(np.float64)
            + aq.x_omega.view(np.float16).astype(np.float64) @ wq.W_omega.view(np.float16).astype(np.float64)
            + L.bias.astype(np.float64))
    np.testing.assert_allclose(y - y0, side, rtol=1e-9, atol=1e-9 * np.max(np.abs(side)))


# ------------------------------------------------------------------ error sanity (monotone)
def test_branches_reduce_quantisation_error_on_outlier_heavy_input():
    """QuantWAMs Fig. 1 / Q-WAM: keeping outlier channels in 16-bit and adding a 16-bit
    low-rank branch lowers the W4A4 error against the unquantised product."""
    errs = []
    for r, n_om in [(0, 0), (0, 32), (32, 32)]:
        L = wlmod.make_layer_inputs("video_dit", M=64, K=512, N=256, rank=r, n_omega=n_om)
        y, *_ = oracle.reference_forward(L)
        ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64) + L.bias
        errs.append(np.linalg.norm(y - ref) / np.linalg.norm(ref))
    assert errs[0] > errs[1] > errs[2], errs
    assert errs[2] < 0.2


# ------------------------------------------------------------------ W8A8
def test_int8_quantiser_rounds_half_even_and_clamps():
    """Per-row int8: scale = amax / 127; every code is the nearest integer of v / scale
    (numpy's round-half-even on the same fp32 quotient) and the largest magnitude is 127."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((16, 256)) * 3).astype(np.float32)
    x[3, :] = 0.0
    bits = wlmod.bf16_bits(x)
    aq = oracle.quantize_act_int8(bits, None, False)
    xf = wlmod.bf16_from_bits(bits)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(aq.scale, (amax / np.float32(127.0)).astype(np.float32))
    for m in range(16):
        if aq.scale[m] == 0:
            assert not aq.q[m].any()
            continue
        t = (xf[m] / aq.scale[m]).astype(np.float32)
        ref = np.clip(np.round(t.astype(np.float64)), -127, 127).astype(np.int8)
        assert np.array_equal(aq.q[m], ref)
        assert np.abs(aq.q[m]).max() == 127


def test_w8a8_plain_case_reduces_to_matmul():
    """s = 1, no rotation: the W8A8 forward equals (qa a)(qw w)^T + b from numpy."""
    L = wlmod.make_layer_inputs("backbone", layer=1, M=10, K=256, N=64, smooth=False, rotate=False)
    y, aq, wq8 = oracle.reference_forward_w8a8(L)
    ref = (aq.q.astype(np.float64) * aq.scale[:, None]) @ (wq8.q.astype(np.float64) * wq8.scale[:, None]).T
    ref += L.bias
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_w8a8_error_is_small_against_unquantised_product():
    """8-bit symmetric quantisation in the smoothed + rotated basis stays within a few
    percent of x W on heavy-tailed inputs (and beats the 4-bit path)."""
    L = wlmod.make_layer_inputs("backbone", layer=1, M=32, K=512, N=128)
    y8, *_ = oracle.reference_forward_w8a8(L)
    y4, *_ = oracle.reference_forward(L)
    ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64) + L.bias
    e8 = np.linalg.norm(y8 - ref) / np.linalg.norm(ref)
    e4 = np.linalg.norm(y4 - ref) / np.linalg.norm(ref)
    assert e8 < 0.02 and e8 < e4, (e8, e4)


# ------------------------------------------------------------------ Conv3d
def _dequant_rows(codes, scales, K):
    return _dequant(codes, scales, K)


def test_conv3d_equals_dequantised_im2col_gemm():
    """The direct convolution equals an explicit numpy im2col of the dequantised voxels times
    the dequantised weight matrix (an independent construction of the same sum)."""
    xb, w = wlmod.make_conv_inputs(T=3, H=5, W=6, C_in=32, C_out=16)
    _, C, D, H, W = xb.shape
    vox = np.arange(D * H * W)
    y, aq, wq = oracle.conv3d_reference(xb, w, vox)
    X = _dequant_rows(aq.codes, aq.scales, C) * np.float64(aq.g[0])           # [V, C]
    Wd = _dequant_rows(wq.codes, wq.scales, 27 * C) * np.float64(wq.gW)      # [N, K]
    Xp = np.zeros((D + 2, H + 2, W + 2, C))
    Xp[1:-1, 1:-1, 1:-1] = X.reshape(D, H, W, C)
    cols = np.stack([Xp[kd:kd + D, kh:kh + H, kw:kw + W].reshape(-1, C)
                     for kd in range(3) for kh in range(3) for kw in range(3)], axis=1).reshape(-1, 27 * C)
    ref = cols @ Wd.T
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10 * np.abs(ref).max())


def test_conv3d_single_voxel_impulse_gives_flipped_kernel():
    """One non-zero input voxel in the middle: each output voxel next to it sees exactly one tap
    (zero padding and the tap order are both exercised)."""
    C, N = 16, 8
    x = np.zeros((1, C, 3, 3, 3), np.float32)
    x[0, :, 1, 1, 1] = np.linspace(1, 2, C, dtype=np.float32)
    w = np.random.default_rng(3).standard_normal((N, C, 3, 3, 3)).astype(np.float32)
    y, aq, wq = oracle.conv3d_reference(wlmod.bf16_bits(x), w, np.arange(27))
    X = _dequant_rows(aq.codes, aq.scales, C) * np.float64(aq.g[0])
    Wd = (_dequant_rows(wq.codes, wq.scales, 27 * C) * np.float64(wq.gW)).reshape(N, 3, 3, 3, C)
    for v in range(27):
        d, h, ww = v // 9, (v // 3) % 3, v % 3
        kd, kh, kw = 1 + 1 - d, 1 + 1 - h, 1 + 1 - ww       # input voxel (1,1,1) = output + k - 1
        ref = Wd[:, kd, kh, kw, :] @ X[13]
        np.testing.assert_allclose(y[v], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


# ------------------------------------------------------------------ 16-bit roundings and side outputs
# Independent single-rounding reference: exact rational arithmetic (fractions.Fraction),
# round-half-even on the integer significand.  Shares nothing with the oracle's C code.
from fractions import Fraction  # noqa: E402


def _round_half_even(q: Fraction) -> int:
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def _exact_bf16_bits(v) -> int:
    """bf16 (8-bit significand, 8-bit exponent, subnormals down to 2^-133) nearest to the
    exact value v (a Fraction or a float), ties to the even significand."""
    neg = (v < 0) if isinstance(v, Fraction) else bool(np.signbit(v))
    sign = 0x8000 if neg else 0
    a = abs(Fraction(v))
    if a == 0:
        return sign
    e = 0                                   # a = m 2^e with m in [1, 2)
    while a >= 2 ** (e + 1):
        e += 1
    while a < Fraction(2) ** e:
        e -= 1
    q = max(e - 7, -133)                    # quantum of the significand (or of a subnormal)
    n = _round_half_even(a / Fraction(2) ** q)
    val = n * Fraction(2) ** q
    if val >= Fraction(2) ** 128:            # beyond the largest finite: infinity
        return sign | 0x7F80
    bits = np.array([float(val)], np.float32).view(np.uint32)[0]
    return sign | int(bits >> 16)


def test_bf16_from_f64_single_rounding_on_values_not_in_fp32():
    """orc_bf16_from_f64 rounds an fp64 value to bf16 ONCE.  The inputs are not fp32
    values, and about half sit just beside a bf16 midpoint, where rounding through fp32
    first (double rounding) gives the wrong neighbour."""
    L = oracle.lib()
    rng = np.random.default_rng(31)
    vals = []
    for _ in range(3000):
        e = int(rng.integers(-120, 120))
        sig = 1 + int(rng.integers(0, 128)) / 128 + 2.0 ** -8     # a bf16 midpoint
        off = float(rng.choice([1, -1])) * 2.0 ** -int(rng.integers(25, 52))
        vals.append(float(rng.choice([1, -1])) * (sig + off) * 2.0 ** e)
    vals += list(rng.standard_normal(3000) * 10.0 ** rng.uniform(-35, 35, 3000))
    vals += [1 + 2 ** -8 + 2 ** -52, 1 + 2 ** -8 - 2 ** -52, 1 + 2 ** -8, 1 + 3 * 2 ** -8,
             2.0 ** -133 * 0.5000001, 2.0 ** -133 * 0.5, 2.0 ** -133 * 1.5, 2.0 ** -140, -0.0]
    assert any(np.float64(np.float32(v)) != v for v in vals)
    bad = [(v, L.orc_bf16_from_f64(v), _exact_bf16_bits(v)) for v in vals
           if L.orc_bf16_from_f64(v) != _exact_bf16_bits(v)]
    assert not bad, bad[:5]
    # the pin distinguishes single from double rounding on these inputs
    double = [v for v in vals if torch.tensor([v], dtype=torch.float64).float().bfloat16().view(torch.uint16).item()
              != _exact_bf16_bits(v)]
    assert len(double) > 500


def test_lowrank_act_equals_exact_product_rounded_once():
    """U = bf16(x P) (Q-WAM abstract, the 16-bit branch's down-projection): against the
    exact rational x P, rounded once to bf16 by the independent routine above.  P is the
    oracle's own bf16(L1 / s) factor, itself checked against torch's conversion."""
    L = wlmod.make_layer_inputs("expert", M=6, K=128, N=32, rank=16)
    wq = oracle.prepare_weights(L.W, L.s, L.L1, L.L2, None, True)
    inv_s = (np.float32(1.0) / L.s).astype(np.float32)
    P_ref = torch.from_numpy((L.L1 * inv_s[:, None]).astype(np.float32)).bfloat16().view(torch.uint16).numpy()
    assert np.array_equal(wq.P, P_ref)
    U = oracle.lowrank_act(L.x_bits, wq.P)
    xf, Pf = wlmod.bf16_from_bits(L.x_bits), wlmod.bf16_from_bits(wq.P)
    for m in range(L.M):
        for j in range(16):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xf[m], Pf[:, j]))
            assert U[m, j] == _exact_bf16_bits(exact), (m, j)


def test_lowrank_act_ties_and_neighbours():
    """Rows built so that x P lands exactly on a bf16 midpoint, or one fp64 ulp beside it:
    the midpoint goes to the even significand, the neighbours go their own way."""
    K = 16
    P = np.zeros((K, 2), np.float32)
    P[:, 0] = 1.0
    P[:3, 1] = [2.0, -1.0, 1.0]
    Pb = wlmod.bf16_bits(P)
    rows = [[1.0, 2.0 ** -8], [1.0, 2.0 ** -8, 2.0 ** -52], [1.0, 2.0 ** -8, -(2.0 ** -52)],
            [1.0, 3 * 2.0 ** -8], [1.0, 3 * 2.0 ** -8, -(2.0 ** -52)], [-3.0, -(2.0 ** -7)]]
    x = np.zeros((len(rows), K), np.float32)
    for i, r in enumerate(rows):
        x[i, :len(r)] = r
    xb = wlmod.bf16_bits(x)
    assert np.array_equal(wlmod.bf16_from_bits(xb), x)          # every entry is a bf16 value
    U = oracle.lowrank_act(xb, Pb)
    want0 = [_exact_bf16_bits(sum(Fraction(float(v)) for v in r)) for r in rows]
    assert U[:, 0].tolist() == want0
    # tie -> even: 1 + 2^-8 -> 1.0; the +ulp neighbour -> 1 + 2^-7; 1 + 3 2^-8 -> 1 + 2^-6
    assert want0[:5] == [0x3F80, 0x3F81, 0x3F80, 0x3F82, 0x3F81]
    want1 = [_exact_bf16_bits(sum(Fraction(float(v)) * Fraction(float(p)) for v, p in zip(x[i], P[:, 1])))
             for i in range(len(rows))]
    assert U[:, 1].tolist() == want1


def test_outlier_slice_values_and_zeroed_codes():
    """x_Omega (QuantWAMs sec. 3.1 Eq. (3), Fig. 1(d)): the fp16 values of the transformed
    channels in Omega, taken before they are zeroed, in Omega's order; those channels then
    quantise to code 0.  Inputs are small integers and powers-of-two smoothing, so the
    block FWHT is exact and equals the dense Sylvester product computed by numpy."""
    rng = np.random.default_rng(41)
    M, K = 5, 256
    x = rng.integers(-900, 900, (M, K)).astype(np.float32)
    x[:, ::7] *= 8                                            # some larger channels
    x = np.clip(x, -255 * 32, 255 * 32)
    xb = wlmod.bf16_bits(x)
    xf = wlmod.bf16_from_bits(xb).astype(np.float64)
    s = (2.0 ** rng.integers(-2, 3, K)).astype(np.float32)
    omega = np.sort(rng.choice(K, 24, replace=False)).astype(np.int32)
    aq = oracle.quantize_act(xb, s, True, omega)
    H = hadamard(64).astype(np.float64) / 8.0
    xt = ((xf / s.astype(np.float64)).reshape(M, K // 64, 64) @ H).reshape(M, K)
    want = xt[:, omega].astype(np.float16).view(np.uint16)
    assert np.array_equal(aq.x_omega, want)
    assert np.any(np.abs(xt[:, omega]) > 2048)                # values that round in fp16
    codes = np.empty((M, K), np.uint8)
    codes[:, 0::2] = aq.codes & 15
    codes[:, 1::2] = aq.codes >> 4
    assert not codes[:, omega].any()                          # kept channels: +0 codes
    kept = np.ones(K, bool)
    kept[omega] = False
    assert codes[:, kept].any()


def test_outlier_slice_on_random_rows_within_one_fp16_ulp():
    """Same pin on Gaussian rows with real smoothing: the fp32 block transform differs from the
    fp64 dense product by a few fp32 ulps, so x_Omega is at most one fp16 ulp from fp16 of the
    dense value and equal to it almost everywhere."""
    L = wlmod.make_layer_inputs("video_dit", M=64, K=512, N=16, rank=0, n_omega=32)
    aq = oracle.quantize_act(L.x_bits, L.s, True, L.omega)
    H = hadamard(64).astype(np.float64) / 8.0
    xs = wlmod.bf16_from_bits(L.x_bits) * (np.float32(1.0) / L.s)
    xt = (xs.astype(np.float64).reshape(64, 8, 64) @ H).reshape(64, 512)
    want = xt[:, L.omega].astype(np.float16)
    got = aq.x_omega.view(np.float16)
    ulp = np.spacing(np.abs(want).astype(np.float16))
    assert np.all(np.abs(got.astype(np.float64) - want.astype(np.float64)) <= ulp.astype(np.float64))
    assert np.mean(got == want) > 0.99


def test_int8_weight_quantiser_against_numpy():
    """Per-output-column int8 of the folded weight (FoldQuantVLA, Key Contribution 3):
    w[n] = fp32(amax_k |Rp[k, n]| / 127); q = clamp(round-half-even(fp32(Rp / w)), +-127)."""
    rng = np.random.default_rng(43)
    K, N = 192, 40
    Rp = (rng.standard_normal((K, N)) * 10 ** rng.uniform(-3, 1, N)[None, :]).astype(np.float32)
    Rp[:, 5] = 0.0
    Rp[:, 7] = np.float32(1.0)
    # entries exactly half-way between two integers after the division
    Rp[::9, 11] = (np.arange(0, K, 9) % 50 + 0.5).astype(np.float32)
    Rp[0, 11] = 127.0
    q = np.zeros((N, K), np.int8)
    w = np.zeros(N, np.float32)
    L = oracle.lib()
    L.orc_quantize_weights_int8(Rp.ctypes.data_as(ctypes.c_void_p), K, N, q.ctypes.data_as(ctypes.c_void_p),
                                w.ctypes.data_as(ctypes.c_void_p))
    w_ref = (np.abs(Rp).max(axis=0) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(w, w_ref)
    with np.errstate(invalid="ignore", divide="ignore"):
        t = (Rp / w_ref[None, :]).astype(np.float32)
    q_ref = np.where(w_ref[None, :] == 0, 0, np.clip(np.round(t.astype(np.float64)), -127, 127)).astype(np.int8).T
    assert np.array_equal(q, q_ref)
    assert q[11, 9] == 10 and q[11, 18] == 18                  # 9.5 -> 10, 18.5 -> 18 (ties to even)
    assert not q[5].any() and np.all(q[7] == 127)


def test_batch_and_fixed_tensor_scales():
    """The two batch-wide tensor-scale modes: per_tensor takes g = amax of the whole batch / 2688;
    a fixed g is used as given (block scales still from each block).  Against closed forms on rows
    whose transform is exact, and against the brute-force block rule of the per-row test."""
    rng = np.random.default_rng(51)
    M, K = 6, 128
    x = rng.integers(-60, 60, (M, K)).astype(np.float32)
    x[2, 5] = 3000.0                                  # the batch maximum (no rotation, s = 1)
    bits = wlmod.bf16_bits(x)
    xf = wlmod.bf16_from_bits(bits)
    per = oracle.quantize_act(bits, None, False, per_tensor=True)
    assert per.g.shape == (1,) and per.g[0] == np.float32(np.float32(np.abs(xf).max()) / np.float32(2688.0))
    # a fixed g equal to the batch's own gives the per-tensor result exactly
    fixed = oracle.quantize_act(bits, None, False, static_g=float(per.g[0]))
    assert np.array_equal(fixed.codes, per.codes) and np.array_equal(fixed.scales, per.scales)
    # a fixed power-of-two g: every block scale is the nearest e4m3 of bmax / 6 / g
    g = np.float32(2.0 ** -3)
    st = oracle.quantize_act(bits, None, False, static_g=float(g))
    assert st.g[0] == g
    sv = np.array([oracle.e4m3_decode(k) for k in range(127)])
    for m in range(M):
        for b in range(K // 16):
            t = np.float32(np.float32(np.abs(xf[m, 16 * b:16 * b + 16]).max()) / np.float32(6.0)) / g
            dist = np.abs(sv - np.float64(t))
            best = np.flatnonzero(dist == dist.min())
            want = 126 if t >= 448 else (best[0] if len(best) == 1 else best[best % 2 == 0][0])
            assert st.scales[m, b] == want
    # saturation: a fixed g far below the data clamps the scale at 448 and the codes at +-6
    sat = oracle.quantize_act(bits, None, False, static_g=1e-6)
    assert sat.scales[2, 0] == 0x7E
    assert (sat.codes[2, 2] & 15) in (7, 15) or (sat.codes[2, 2] >> 4) in (7, 15)


# ------------------------------------------------------------------ the rotate-then-smooth order
@pytest.mark.parametrize("r,n_om", [(0, 0), (16, 0), (0, 16), (16, 16)])
def test_folding_invariance_rotate_then_smooth(r, n_om):
    """QuantWAMs sec. 3.1 Eq. (1) order, A R S^-1 (rotation first): with quantisation disabled
    the folded graph x H S^-1 . S H (W - P Q) + x P Q (+ outliers) still computes x W + b
    (FoldQuantVLA Proposition 1 in this order)."""
    L = wlmod.make_layer_inputs("tiny", M=8, K=256, N=96, rank=r, n_omega=n_om, smooth_after=True)
    with oracle.transform_order(True):
        wq = oracle.prepare_weights(L.W, L.s, L.L1, L.L2, L.omega, True)
    y = oracle.forward_noquant(L.x_bits, L.s, True, L.omega, wq, L.bias, smooth_after=True)
    ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64)
    if L.bias is not None:
        ref += L.bias
    assert np.max(np.abs(y - ref)) / np.max(np.abs(ref)) <= 1e-5


def test_rotate_then_smooth_transform_against_dense_matrices():
    """The activation transform in this order equals (x H) diag(1/s) from dense fp64 matrices on
    integer rows with power-of-two smoothing (exact in fp32), and differs from the default order
    there; P = bf16(H S^-1 L1) matches the dense product rounded once."""
    rng = np.random.default_rng(61)
    M, K = 4, 128
    x = rng.integers(-500, 500, (M, K)).astype(np.float32)
    bits = wlmod.bf16_bits(x)
    s = (2.0 ** rng.integers(-2, 3, K)).astype(np.float32)
    with oracle.transform_order(True):
        aq = oracle.quantize_act(bits, s, True, keep_xt=True)
    H = hadamard(64).astype(np.float64) / 8.0
    xf = wlmod.bf16_from_bits(bits).astype(np.float64)
    want = (xf.reshape(M, 2, 64) @ H).reshape(M, K) / s.astype(np.float64)
    assert np.array_equal(aq.xt.astype(np.float64), want)
    other = oracle.quantize_act(bits, s, True, keep_xt=True)
    assert not np.array_equal(other.xt, aq.xt)
    L1 = rng.standard_normal((K, 8)).astype(np.float32)
    L2 = rng.standard_normal((8, 32)).astype(np.float32)
    W = rng.standard_normal((K, 32)).astype(np.float32)
    with oracle.transform_order(True):
        wq = oracle.prepare_weights(W, s, L1, L2, None, True)
    inv_s = (np.float32(1.0) / s).astype(np.float64)
    Pd = (H @ (inv_s[:, None] * L1.astype(np.float64)).reshape(2, 64, 8)).reshape(K, 8)
    assert np.array_equal(wq.P, np.array([[_exact_bf16_bits(float(v)) for v in row] for row in Pd], np.uint16))


# ------------------------------------------------------------------ FP8 W8A8
def test_signed_e4m3_against_torch_float8():
    """Signed e4m3 (sign bit 7): against torch's fp32 -> float8_e4m3fn conversion (round to nearest
    even) on finite values within range, both signs, and saturation to +-448 above it."""
    rng = np.random.default_rng(71)
    v = np.concatenate([rng.uniform(-448, 448, 100000), np.sign(rng.standard_normal(100000)) *
                        2.0 ** rng.uniform(-12, 8.8, 100000)]).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    L = oracle.lib()
    got = np.array([L.orc_e4m3s_encode(float(a)) for a in v[:30000]], np.uint8)
    assert np.array_equal(got, ref[:30000])
    assert L.orc_e4m3s_encode(1e6) == 0x7E and L.orc_e4m3s_encode(-1e6) == 0xFE
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert L.orc_e4m3s_decode(c) == float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float())


def test_fp8_quantiser_rule_against_numpy_and_torch():
    """Per-row FP8: scale = fp32(amax / 448); codes = e4m3(fp32(v / scale)) -- the quotient from numpy,
    the rounding to e4m3 from torch; the row maximum maps to +-448."""
    rng = np.random.default_rng(72)
    x = (rng.standard_normal((12, 256)) * 3).astype(np.float32)
    x[5, :] = 0.0
    bits = wlmod.bf16_bits(x)
    aq = oracle.quantize_act_fp8(bits, None, False)
    xf = wlmod.bf16_from_bits(bits)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(aq.scale, (amax / np.float32(448.0)).astype(np.float32))
    for m in range(12):
        if aq.scale[m] == 0:
            assert not aq.q[m].any()
            continue
        t = (xf[m] / aq.scale[m]).astype(np.float32)
        ref = torch.from_numpy(np.clip(t, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(aq.q[m], ref)
        assert (aq.q[m] & 0x7F).max() == 0x7E


def test_fp8_w8a8_plain_case_reduces_to_matmul_and_beats_w4a4():
    """s = 1, no rotation: the FP8 forward equals (dec(qa) a)(dec(qw) w)^T + b from numpy (decoding by
    torch); in the smoothed + rotated basis its error against x W is below the 4-bit path's."""
    L = wlmod.make_layer_inputs("backbone", layer=1, M=10, K=256, N=64, smooth=False, rotate=False)
    y, aq, wq8 = oracle.reference_forward_fp8(L)
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    ref = (dec(aq.q) * aq.scale[:, None]) @ (dec(wq8.q) * wq8.scale[:, None]).T + L.bias
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    L = wlmod.make_layer_inputs("backbone", layer=1, M=32, K=512, N=128)
    y8, *_ = oracle.reference_forward_fp8(L)
    y4, *_ = oracle.reference_forward(L)
    ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64) + L.bias
    e8 = np.linalg.norm(y8 - ref) / np.linalg.norm(ref)
    e4 = np.linalg.norm(y4 - ref) / np.linalg.norm(ref)
    assert e8 < 0.05 and e8 < e4, (e8, e4)


# ------------------------------------------------------------------ outlier calibration
@pytest.mark.parametrize("after", [False, True])
def test_pooled_energy_against_dense_transform(after):
    """z(c) = mean_t xt[t,c]^2 (QuantWAMs sec. 3.1 Eq. (1)-(3), one context): on integer rows with
    power-of-two smoothing the fp32 transform is exact, so z equals numpy's fp64 mean of the dense
    Sylvester product squared (up to fp64 summation); random rows within 1e-6 of it."""
    rng = np.random.default_rng(81)
    M, K = 37, 192
    x = rng.integers(-300, 300, (M, K)).astype(np.float32)
    bits = wlmod.bf16_bits(x)
    s = (2.0 ** rng.integers(-2, 3, K)).astype(np.float32)
    H = hadamard(64).astype(np.float64) / 8.0
    xf = wlmod.bf16_from_bits(bits).astype(np.float64)
    inv = 1.0 / s.astype(np.float64)
    if after:
        xt = (xf.reshape(M, 3, 64) @ H).reshape(M, K) * inv
    else:
        xt = ((xf * inv).reshape(M, 3, 64) @ H).reshape(M, K)
    want = (xt * xt).mean(axis=0)
    got = oracle.pooled_energy(bits, s, True, after)
    np.testing.assert_allclose(got, want, rtol=1e-14)
    L = wlmod.make_layer_inputs("video_dit", M=64, K=256, N=16, rank=0, n_omega=0)
    sm = L.s
    xs = wlmod.bf16_from_bits(L.x_bits).astype(np.float64) / sm.astype(np.float64)
    xt = (xs.reshape(64, 4, 64) @ H).reshape(64, 256)
    np.testing.assert_allclose(oracle.pooled_energy(L.x_bits, sm, True), (xt * xt).mean(axis=0), rtol=1e-6)


def test_topk_channels_ties_and_order():
    z = np.array([1.0, 5.0, 3.0, 5.0, 0.5, 3.0, 7.0, 5.0])
    assert oracle.topk_channels(z, 3).tolist() == [1, 3, 6]         # 7, then the two lowest 5s
    assert oracle.topk_channels(z, 5).tolist() == [1, 2, 3, 6, 7]
    assert oracle.topk_channels(z, 0).tolist() == []
    rng = np.random.default_rng(82)
    z = rng.standard_normal(1000) ** 2
    want = np.sort(np.lexsort((np.arange(1000), -z))[:41])
    assert np.array_equal(oracle.topk_channels(z, 41), want)


# ------------------------------------------------------------------ W4A8 (A8-protected steps)
def test_w4a8_reduces_to_dequantised_matmul_and_sits_between_w4a4_and_fp8():
    """s = 1, no rotation, no branches: the W4A8 forward equals (dec(qa) a)(deq(W) gW)^T + b from
    numpy with torch decoding the e4m3 codes; with branches and transforms its error lies below the
    W4A4 error (8-bit activations) on the same 4-bit weights; kept channels leave the e4m3 codes at 0."""
    L = wlmod.make_layer_inputs("expert", M=9, K=256, N=48, rank=0, n_omega=0, smooth=False, rotate=False)
    y, aq, wq, _ = oracle.reference_forward_w4a8(L)
    dec = torch.from_numpy(aq.q).view(torch.float8_e4m3fn).double().numpy()
    B = _dequant(wq.codes, wq.scales, 256) * np.float64(wq.gW)
    ref = (dec * aq.scale[:, None].astype(np.float64)) @ B.T + L.bias
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    L = wlmod.make_layer_inputs("video_dit", M=48, K=512, N=128, rank=16, n_omega=16)
    y8, a8, *_ = oracle.reference_forward_w4a8(L)
    y4, *_ = oracle.reference_forward(L)
    ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64) + L.bias
    e8 = np.linalg.norm(y8 - ref) / np.linalg.norm(ref)
    e4 = np.linalg.norm(y4 - ref) / np.linalg.norm(ref)
    assert e8 < e4, (e8, e4)
    assert not a8.q[:, L.omega].any()
    aq4 = oracle.quantize_act(L.x_bits, L.s, True, L.omega)
    assert np.array_equal(a8.x_omega, aq4.x_omega)            # the same fp16 kept channels


# ------------------------------------------------------------------ Q-WAM projected complement
def test_projected_complement_is_orthogonal_and_keeps_the_fold():
    """Q-WAM abstract (the complementary activations are quantised): xt_c = xt - u Vt is (up to the
    bf16 roundings of u and Vt) orthogonal to the protected subspace, and with quantisation off the
    three branches still compute x W + b (x_c R = x_s R for the complement R)."""
    L = wlmod.make_layer_inputs("video_dit", M=24, K=256, N=64, rank=16, n_omega=0)
    wq = oracle.prepare_weights(L.W, L.s, L.L1, L.L2, None, True)
    U = oracle.lowrank_act(L.x_bits, wq.P)
    Vt = oracle.projection_basis(L.L1, True)
    aq = oracle.quantize_act_projected(L.x_bits, L.s, True, None, U, Vt, keep_xt=True)
    H = hadamard(64).astype(np.float64) / 8.0
    Ur = L.L1.astype(np.float64) / np.linalg.norm(L.L1.astype(np.float64), axis=0)[None, :]
    HUr = (H @ Ur.reshape(4, 64, 16)).reshape(256, 16)          # the subspace in the rotated basis
    xt = oracle.quantize_act(L.x_bits, L.s, True, keep_xt=True).xt.astype(np.float64)
    before = np.abs(xt @ HUr).max()
    after = np.abs(aq.xt.astype(np.float64) @ HUr).max()
    assert after < 1e-2 * before, (before, after)
    # the fold: xt_c R' + u Q + b = x W + b without quantisation
    y = aq.xt.astype(np.float64) @ wq.Rp.astype(np.float64) + \
        wlmod.bf16_from_bits(U).astype(np.float64) @ wlmod.bf16_from_bits(wq.Q).astype(np.float64) + L.bias
    ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64) + L.bias
    assert np.max(np.abs(y - ref)) / np.max(np.abs(ref)) < 2e-2
    ynp = xt @ wq.Rp.astype(np.float64) + wlmod.bf16_from_bits(U).astype(np.float64) @ \
        wlmod.bf16_from_bits(wq.Q).astype(np.float64) + L.bias
    assert np.max(np.abs(y - ynp)) / np.max(np.abs(ref)) < 2e-2


def test_projection_basis_and_fma_sequence_against_numpy():
    """Vt = bf16(S^-2 L1^T H) from dense fp64 matrices (single rounding); the subtraction is the fp32
    fma sequence j = 0 .. r-1, restated with numpy's fp32 arithmetic via the exact fp64 product."""
    rng = np.random.default_rng(91)
    K, r = 128, 8
    L1 = rng.standard_normal((K, r)).astype(np.float32)
    Vt = oracle.projection_basis(L1, True)
    H = hadamard(64).astype(np.float64) / 8.0
    l1 = L1.astype(np.float64)
    want = ((H @ l1.reshape(2, 64, r)).reshape(K, r) / (l1 * l1).sum(axis=0)[None, :]).T
    assert np.array_equal(Vt, np.array([[_exact_bf16_bits(float(v)) for v in row] for row in want], np.uint16))
    M = 5
    x = rng.standard_normal((M, K)).astype(np.float32)
    u = wlmod.bf16_bits(rng.standard_normal((M, r)).astype(np.float32))
    xt = x.copy()
    oracle.lib().orc_project_complement(xt.ctypes.data_as(ctypes.c_void_p), M, K, u.ctypes.data_as(ctypes.c_void_p),
                                        Vt.ctypes.data_as(ctypes.c_void_p), r)
    uf = wlmod.bf16_from_bits(u).astype(np.float64)
    vf = wlmod.bf16_from_bits(Vt).astype(np.float64)
    acc = x.copy()
    for j in range(r):      # fma: the exact product and sum rounded once to fp32
        acc = (acc.astype(np.float64) - uf[:, j:j + 1] * vf[j][None, :]).astype(np.float32)
    assert np.array_equal(xt, acc)


def test_projected_complement_lowers_error_when_the_subspace_carries_the_outliers():
    """When the activations' large components lie in the protected subspace, quantising the
    complement instead of the whole activation lowers the W4A4 error (Q-WAM's premise)."""
    L = wlmod.make_layer_inputs("video_dit", M=64, K=512, N=128, rank=16, n_omega=0)
    rng = np.random.default_rng(92)
    s = L.s.astype(np.float64)
    Ur = L.L1.astype(np.float64) / np.linalg.norm(L.L1.astype(np.float64), axis=0)[None, :]
    x = L.x_f32.astype(np.float64) + 20.0 * (rng.standard_normal((64, 16)) @ Ur.T) * s[None, :]
    L.x_bits = wlmod.bf16_bits(x.astype(np.float32))
    y_p, *_ = oracle.reference_forward_projected(L)
    y_n, *_ = oracle.reference_forward(L)
    ref = L.x_f32.astype(np.float64) @ L.W.astype(np.float64) + L.bias
    e_p = np.linalg.norm(y_p - ref) / np.linalg.norm(ref)
    e_n = np.linalg.norm(y_n - ref) / np.linalg.norm(ref)
    assert e_p < e_n, (e_p, e_n)
