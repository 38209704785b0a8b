"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar (written here, derived in the design notes):
  * weight and activation codes, e4m3 scales, fp32 row/tensor scales, fp16 outlier
    values: bit-exact;
  * U = bf16(x P): within one bf16 ulp plus the fp32 summation bound K 2^-24 sum|x P|
    (fp32 vs fp64 accumulation before one rounding);
  * y: |y_gpu - y_oracle| <= 1e-3 (|y| + ||x_row|| ||w_col|| / sqrt(K)) + 2^-8 |y|
    (fp32 accumulation vs fp64, plus the bf16 rounding of the output), plus, where the oracle's U
    is at hand, U's bound above carried through Q (sum_j dU_j |Q_jn|): a U element within one
    bf16 ulp of the oracle's moves y by that much.
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


def x_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def prep(L, **kw):
    return wq.wq_prepare_weights(L.spec.K, L.spec.N, L.W, L.bias, L.s, L.L1, L.L2,
                                 L.omega if L.omega.size else None, rotate=L.rotate,
                                 transform_order=int(L.smooth_after), **kw)


def oq(L, **kw):
    """The oracle's activation quantiser in the layer's transform order."""
    with oracle.transform_order(L.smooth_after):
        return oracle.quantize_act(L.x_bits, L.s, L.rotate, L.omega, **kw)


def ow(L):
    """The oracle's weight fold and quantiser in the layer's transform order."""
    with oracle.transform_order(L.smooth_after):
        return oracle.prepare_weights(L.W, L.s, L.L1, L.L2, L.omega, L.rotate)


def y_tolerance(L, y_ref, rows=None):
    x = L.x_f32 if rows is None else L.x_f32[rows]
    xn = np.linalg.norm(x.astype(np.float64), axis=1)[:, None]
    wn = np.linalg.norm(L.W.astype(np.float64), axis=0)[None, :]
    return 1e-3 * (np.abs(y_ref) + xn * wn / np.sqrt(L.spec.K)) + 2.0 ** -8 * np.abs(y_ref)


def u_term(L, ref, rows=None):
    """The part of y's bound that U's own bound (u_close: one bf16 ulp plus the fp32 summation
    bound, fp32 on the device vs fp64 in the oracle) contributes through Q: sum_j dU[m, j] |Q[j, n]|."""
    _, _, o, U = ref
    if U is None or not L.rank:
        return 0.0
    xb = L.x_bits if rows is None else L.x_bits[rows]
    b = np.abs(wl.bf16_from_bits(U).astype(np.float64))
    absdot = np.abs(wl.bf16_from_bits(xb).astype(np.float64)) @ np.abs(wl.bf16_from_bits(o.P).astype(np.float64))
    dU = np.maximum(b * 2.0 ** -7, 2.0 ** -133) + L.spec.K * 2.0 ** -24 * absdot
    return dU @ np.abs(wl.bf16_from_bits(o.Q).astype(np.float64))


def assert_y_close(L, y_gpu, y_ref, rows=None, ref=None):
    """y within y_tolerance; with the oracle's full result `ref` (reference_forward's tuple) the
    bound also carries U's bound through Q."""
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    tol = y_tolerance(L, y_ref, rows)
    if ref is not None:
        tol = tol + u_term(L, ref, rows)
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside tolerance; worst excess "
                           f"{np.max(err - tol):.3g} at {np.unravel_index(np.argmax(err - tol), err.shape)}")
    return float(np.max(err / np.maximum(tol, 1e-30)))


def u_close(u_gpu_bits, u_ref_bits, x_bits, P_bits):
    """U = bf16(x P): the GPU sums in fp32, the oracle in fp64, each then rounds once.
    Bound: one bf16 ulp of the reference plus the fp32 summation bound K 2^-24 sum|x P|."""
    a = wl.bf16_from_bits(u_gpu_bits).astype(np.float64)
    b = wl.bf16_from_bits(u_ref_bits).astype(np.float64)
    K = x_bits.shape[1]
    absdot = np.abs(wl.bf16_from_bits(x_bits).astype(np.float64)) @ np.abs(
        wl.bf16_from_bits(P_bits).astype(np.float64))
    ulp = np.maximum(np.abs(b) * 2.0 ** -7, 2.0 ** -133)
    return np.abs(a - b) <= ulp + K * 2.0 ** -24 * absdot


CASES = {
    "tiny_full": ("tiny", dict()),
    "expert_small": ("expert", dict(M=50, K=1024, N=512)),
    "ragged_m130": ("expert", dict(M=130, K=256, N=384, rank=16)),
    "dit_r32_o64_ragged_n": ("video_dit", dict(M=200, K=512, N=272, rank=32, n_omega=64)),
    "backbone_r0": ("backbone", dict(layer=0, M=129, K=2048, N=256)),
    "no_rotate_o16": ("video_dit", dict(M=64, K=1536, N=128, rank=32, n_omega=16, rotate=False)),
    "no_smooth_r64": ("expert", dict(M=33, K=640, N=160, rank=64, smooth=False)),
    "min_k64_n16_m1": ("expert", dict(M=1, K=64, N=16, rank=0)),
    "multi_tile_kstage_tail": ("expert", dict(M=260, K=1088, N=400, rank=16)),
    # QuantWAMs sec. 4.2 keeps the top 2% of the input channels: 41 of 2048; ranks that are not
    # a side-MMA width (stored zero-padded to 16 / 32 / 64)
    "top2pct_o41_r24": ("video_dit", dict(M=96, K=2048, N=256, rank=24, n_omega=41)),
    "o5_r8": ("video_dit", dict(M=40, K=512, N=192, rank=8, n_omega=5)),
    "o64_r40_no_rotate": ("video_dit", dict(M=150, K=1024, N=144, rank=40, n_omega=64, rotate=False)),
    # rotation first, then smoothing (QuantWAMs sec. 3.1 Eq. (1), A R S^-1)
    "rot_smooth_r32_o16": ("video_dit", dict(M=96, K=1024, N=192, rank=32, n_omega=16, smooth_after=True)),
    "rot_smooth_expert_r32": ("expert", dict(M=50, K=1024, N=256, rank=32, smooth_after=True)),
}


def side_out(t, count):
    """The first `count` columns of a strided side output, and its padding (must be zero)."""
    a = t.cpu().view(torch.int16).numpy().view(np.uint16)
    return a[:, :count], a[:, count:]


def layer(case):
    name, kw = CASES[case]
    return wl.make_layer_inputs(name, **kw)


@pytest.mark.parametrize("case", list(CASES))
def test_weights_bitexact(case):
    L = layer(case)
    w = prep(L)
    ex = wq.wq_export_weights(w)
    o = ow(L)
    assert np.float32(ex["gW"]) == np.float32(o.gW)
    assert np.array_equal(ex["scales"], o.scales)
    assert np.array_equal(ex["codes"], o.codes)
    assert np.array_equal(ex["P"], o.P) and np.array_equal(ex["Q"], o.Q)
    assert np.array_equal(ex["W_omega"], o.W_omega)


@pytest.mark.parametrize("case", list(CASES))
def test_activation_quant_bitexact(case):
    L = layer(case)
    w = prep(L)
    x = x_dev(L.x_bits)
    codes, scales, g, xo, u = wq.wq_quantize_activations(w, x, wq.WQ_SCALE_LAYOUT_ROWMAJOR)
    codes2, sf_mma, g2, _, _ = wq.wq_quantize_activations(w, x, wq.WQ_SCALE_LAYOUT_MMA)
    torch.cuda.synchronize()
    aq = oq(L)
    assert np.array_equal(g.cpu().numpy(), aq.g)
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    M, K = L.x_bits.shape
    assert np.array_equal(wq.mma_scales_to_rowmajor(sf_mma.cpu().numpy(), M, K), aq.scales)
    assert np.array_equal(codes2.cpu().numpy(), aq.codes) and np.array_equal(g2.cpu().numpy(), aq.g)
    check_side(L, xo, u, aq)


def check_side(L, xo, u, aq):
    """x_Omega bit-exact and U within its bound, in their strided layouts (padding zero)."""
    if L.omega.size:
        got, pad = side_out(xo, L.omega.size)
        assert np.array_equal(got, aq.x_omega) and not pad.any()
    if L.rank:
        o = ow(L)
        U = oracle.lowrank_act(L.x_bits, o.P)
        ug, pad = side_out(u, L.rank)
        assert u_close(ug, U, L.x_bits, o.P).all() and not pad.any()


@pytest.mark.parametrize("case,split", [("expert_small", 1), ("expert_small", 4), ("expert_small", 16),
                                        ("dit_r32_o64_ragged_n", 2), ("dit_r32_o64_ragged_n", 3),
                                        ("dit_r32_o64_ragged_n", 8), ("no_smooth_r64", 1), ("no_smooth_r64", 5),
                                        ("backbone_r0", 2), ("multi_tile_kstage_tail", 3),
                                        ("multi_tile_kstage_tail", 16)])
def test_activation_quant_split(case, split, tuning):
    """The quantiser with a row tile's K range on one CTA or spread over a cluster of 2..16
    CTAs, including sizes that split the blocks unevenly (the row amax and the low-rank
    partial sums then go through distributed shared memory)."""
    tuning("WQ_QUANT_SPLIT", str(split))
    L = layer(case)
    w = prep(L)
    x = x_dev(L.x_bits)
    codes, scales, g, xo, u = wq.wq_quantize_activations(w, x, wq.WQ_SCALE_LAYOUT_ROWMAJOR)
    torch.cuda.synchronize()
    aq = oq(L)
    assert np.array_equal(g.cpu().numpy(), aq.g)
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    check_side(L, xo, u, aq)


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("schedule", ["stream", "cluster", "resident"])
def test_activation_quant_schedules(case, schedule, tuning):
    """Every quantiser schedule on every case: persistent CTAs that stream each row tile's
    blocks twice (the second pass recomputes the transform), clusters that keep the transformed
    blocks resident in shared memory, and persistent CTAs (clusters for a wide K) that keep each
    row tile's transformed values in registers."""
    tuning("WQ_QUANT_SCHEDULE", schedule)
    L = layer(case)
    w = prep(L)
    x = x_dev(L.x_bits)
    codes, scales, g, xo, u = wq.wq_quantize_activations(w, x, wq.WQ_SCALE_LAYOUT_MMA)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w)
    aq = oq(L)
    assert np.array_equal(g.cpu().numpy(), aq.g)
    assert np.array_equal(wq.mma_scales_to_rowmajor(scales.cpu().numpy(), L.M, L.spec.K), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    check_side(L, xo, u, aq)


@pytest.mark.parametrize("case", list(CASES))
def test_forward_parity(case):
    L = layer(case)
    w = prep(L)
    y = wq.wq_linear_forward(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    ref = oracle.reference_forward(L)
    y_ref = ref[0]
    assert_y_close(L, y, y_ref, ref=ref)


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("fused", ["1", "0"])
def test_forward_parity_fused_and_two_kernel_paths(case, fused, tuning):
    """With WQ_FUSED=1, small batches (M <= 64, rank <= 32, K % 128 == 0) run quantiser and
    GEMM fused in one cluster kernel (codes built in shared memory, row maxima and U partials
    across the cluster, split-K partials summed in rank order); WQ_FUSED=0 keeps the
    two-kernel path on the same case.  The path actually taken is checked first."""
    tuning("WQ_FUSED", fused)
    L = layer(case)
    w = prep(L)
    eligible = L.M <= 64 and L.rank <= 32 and L.spec.K % 128 == 0 and not L.smooth_after
    expected = wq.WQ_PATH_FUSED if fused == "1" and eligible else wq.WQ_PATH_TWO_KERNEL
    assert wq.wq_forward_path(w, L.M) == expected
    y = wq.wq_linear_forward(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    ref = oracle.reference_forward(L)
    y_ref = ref[0]
    assert_y_close(L, y, y_ref, ref=ref)


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("wide", ["db", "1", "0"])
def test_forward_parity_gemm_schedules(case, wide, tuning):
    """Every GEMM schedule on every case: 256 x 192 tiles on CTA pairs with two accumulators
    ("db": the side branch of one tile computed while the next tile's main loop runs), 256 x 256
    tiles on CTA pairs (tcgen05 cta_group::2, single-buffered accumulator, side branch computed
    into the drained accumulator) and 128 x 128 tiles on single CTAs; partial tiles in M and N
    included."""
    tuning("WQ_GEMM_WIDE", "0" if wide == "0" else "1")
    tuning("WQ_GEMM_DB", "1" if wide == "db" else "0")
    tuning("WQ_FUSED", "0")              # small batches too run the GEMM under test
    L = layer(case)
    w = prep(L)
    sched = wq.wq_gemm_schedule(w, L.M)
    assert sched == {"db": wq.WQ_GEMM_WIDE_DB, "1": wq.WQ_GEMM_WIDE}.get(wide, sched)
    assert (sched in (wq.WQ_GEMM_WIDE, wq.WQ_GEMM_WIDE_DB)) == (wide != "0")
    y = wq.wq_linear_forward(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    ref = oracle.reference_forward(L)
    y_ref = ref[0]
    assert_y_close(L, y, y_ref, ref=ref)


@pytest.mark.parametrize("case,split", [("expert_small", 1), ("expert_small", 2), ("expert_small", 4),
                                        ("multi_tile_kstage_tail", 1), ("multi_tile_kstage_tail", 2),
                                        ("multi_tile_kstage_tail", 4), ("dit_r32_o64_ragged_n", 2),
                                        ("backbone_r0", 8), ("no_smooth_r64", 2), ("min_k64_n16_m1", 1)])
@pytest.mark.parametrize("push", ["1", "0"])
def test_forward_parity_split_k(case, split, push, tuning):
    """Both GEMM schedules: one persistent CTA per tile (split 1) and the K range of a tile
    spread over a cluster (split > 1), its rank-ordered reduction in both forms: partial rows
    pushed into the reducing rank's shared memory, or pulled from every peer."""
    tuning("WQ_GEMM_SPLIT", str(split))
    tuning("WQ_GEMM_PUSH", push)
    tuning("WQ_FUSED", "0")
    L = layer(case)
    w = prep(L)
    y = wq.wq_linear_forward(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    ref = oracle.reference_forward(L)
    y_ref = ref[0]
    assert_y_close(L, y, y_ref, ref=ref)


def test_forward_is_deterministic_and_host_path_matches():
    L = layer("dit_r32_o64_ragged_n")
    w = prep(L)
    x = x_dev(L.x_bits)
    y1 = wq.wq_linear_forward(w, x)
    y2 = wq.wq_linear_forward(w, x)
    codes, sf, g, xo, u = wq.wq_quantize_activations(w, x, wq.WQ_SCALE_LAYOUT_MMA)
    y3 = wq.wq_linear_forward_quantized(w, codes, sf, g, u, xo)
    M = x.shape[0]
    xh = x.cpu().pin_memory()
    yh = torch.empty((M, L.spec.N), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(wq.wq_host_workspace_bytes(w, M), dtype=torch.uint8, device="cuda")
    wq.wq_linear_forward_host(w, xh, yh, ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert torch.equal(y1, y3)
    assert torch.equal(y1.cpu(), yh)


@pytest.mark.parametrize("M", [4100, 16384])
def test_host_path_row_chunks(M):
    """From 4096 rows the host-buffer path runs in row chunks with the uploads and downloads on the
    handle's copy streams; on a side stream that alone is synchronised, y equals the device path
    run on the same chunks, bit for bit, and the oracle on sampled rows within tolerance."""
    L = wl.make_layer_inputs("video_dit", M=M, K=512, N=272, rank=32, n_omega=16)
    w = prep(L)
    x = x_dev(L.x_bits)
    nch = max(1, min(8, M // 2048))
    per = -(-(-(-M // nch)) // 256) * 256
    y_dev = torch.cat([wq.wq_linear_forward(w, x[r0:r0 + per]) for r0 in range(0, M, per)])
    xh = x.cpu().pin_memory()
    yh = torch.zeros((M, L.spec.N), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(wq.wq_host_workspace_bytes(w, M), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    wq.wq_linear_forward_host(w, xh, yh, ws, side)
    side.synchronize()
    wq.wq_check_device_error(w)
    assert torch.equal(y_dev.cpu(), yh)
    rows = _sampled_rows(M, 24, 7)
    ref = oracle.reference_forward(L, rows=rows)
    assert_y_close(L, yh[torch.from_numpy(rows)], ref[0], rows, ref=ref)


def test_zero_rows_and_empty_batch():
    L = wl.make_layer_inputs("expert", M=40, K=256, N=128, rank=16)
    bits = L.x_bits.copy()
    bits[3] = 0
    bits[17] = 0x8000            # -0.0 everywhere
    L.x_bits = bits
    w = prep(L)
    y = wq.wq_linear_forward(w, x_dev(bits))
    _, _, g, _, _ = wq.wq_quantize_activations(w, x_dev(bits))
    torch.cuda.synchronize()
    assert g[3].item() == 0.0 and g[17].item() == 0.0
    ref = oracle.reference_forward(L)
    y_ref = ref[0]
    assert_y_close(L, y, y_ref, ref=ref)
    empty = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    y0 = wq.wq_linear_forward(w, empty)
    assert y0.shape == (0, 128)


def test_rounding_ties_through_the_quantiser():
    """With s = 1 and no rotation the quantiser sees x itself.  A row holding 2688 has
    g = 1 exactly; blocks with maximum 6 * 2^j get scale 2^j, so the other values sit
    exactly on e2m1 midpoints, on grid points, just beside them, and at +-0."""
    K = 256
    rows = []
    # midpoints, grid points, one bf16 step either side of a midpoint, above-max values
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 3.0, 4.0, 0.2490234375, 1.2578125, 5.5, 7.0]
    for j in range(-3, 4):
        r = np.zeros(K, np.float32)
        r[0] = 2688.0
        for b in range(1, K // 16):
            blk = np.array(mids + [6.0], np.float32) * np.float32(2.0 ** j)
            blk *= np.where(np.arange(16) % 2 == (b % 2), -1.0, 1.0).astype(np.float32)
            r[16 * b:16 * b + 16] = blk
        r[17] = -0.0
        r[18] = 0.0
        rows.append(r)
    x = np.stack(rows)
    bits = wl.bf16_bits(x)
    assert np.array_equal(wl.bf16_from_bits(bits), x)
    W = np.random.default_rng(0).standard_normal((K, 64)).astype(np.float32) * 0.02
    w = wq.wq_prepare_weights(K, 64, W, rotate=False)
    codes, scales, g, _, _ = wq.wq_quantize_activations(w, x_dev(bits))
    torch.cuda.synchronize()
    aq = oracle.quantize_act(bits, None, False)
    assert np.all(aq.g == 1.0)
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)


def _e4m3_midpoints():
    """Every midpoint between neighbouring positive e4m3 values (subnormal and normal)."""
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue                      # NaN
            vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    vals = sorted(set(vals))
    return [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]


@pytest.mark.parametrize("schedule", ["stream", "cluster"])
def test_scale_ties_through_the_quantiser(schedule, tuning):
    """Block maxima at 6 x every e4m3 midpoint (and one bf16 step either side) in rows with
    g = 1: (bmax / 6) / g lands exactly on the scale's rounding boundaries, where the fast
    reciprocal path has to hand over to the exact divisions."""
    tuning("WQ_QUANT_SCHEDULE", schedule)
    K = 512
    targets = []
    for mid in _e4m3_midpoints():
        v = np.float32(6.0 * mid)
        b = int(wl.bf16_bits(np.array([v], np.float32))[0])
        for d in (-1, 0, 1):
            targets.append(float(wl.bf16_from_bits(np.array([b + d], np.uint16))[0]))
    per_row = K // 16 - 1
    rows = []
    for i in range(0, len(targets), per_row):
        r = np.zeros(K, np.float32)
        r[0] = 2688.0
        for j, t in enumerate(targets[i:i + per_row]):
            blk = np.linspace(0.0, t, 16, dtype=np.float32)
            blk[-1] = t
            r[16 * (j + 1):16 * (j + 2)] = wl.bf16_from_bits(wl.bf16_bits(blk))
        rows.append(r)
    x = np.stack(rows)
    bits = wl.bf16_bits(x)
    W = np.random.default_rng(1).standard_normal((K, 32)).astype(np.float32) * 0.02
    w = wq.wq_prepare_weights(K, 32, W, rotate=False)
    codes, scales, g, _, _ = wq.wq_quantize_activations(w, x_dev(bits))
    torch.cuda.synchronize()
    aq = oracle.quantize_act(bits, None, False)
    assert np.all(aq.g == 1.0)
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)


# ------------------------------------------------------------------ full sizes
def _sampled_rows(M, n, seed):
    return np.sort(np.random.default_rng(seed).choice(M, size=n, replace=False))


def _tile_rows(M, seed):
    """One row in every 128-row GEMM tile (a seeded position inside it), the first and the last
    row of the batch, and the last row of each 256-row pair tile."""
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    for t in range(0, M, 128):
        rows.add(t + int(rng.integers(0, min(128, M - t))))
    for t in range(255, M, 256):
        rows.add(t)
    return np.array(sorted(rows))


@pytest.mark.parametrize("layer_idx", [0, 1])
def test_expert_batch1_full_size(layer_idx):
    L = wl.make_layer_inputs("expert", layer=layer_idx)
    w = prep(L)
    y = wq.wq_linear_forward(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    ref = oracle.reference_forward(L)
    y_ref = ref[0]
    assert_y_close(L, y, y_ref, ref=ref)


@pytest.mark.parametrize("wl_name,layer_idx", [("video_dit", 0), ("video_dit", 1), ("video_dit", 2),
                                               ("video_dit", 3), ("backbone", 0), ("backbone", 2)])
def test_full_size_every_row_and_tile(wl_name, layer_idx):
    """Full workload sizes in the launch configuration the benchmark times: codes, scales, row
    scales and x_Omega of EVERY row bit-exact against the oracle's quantiser (both quantiser
    schedules agree with it), and y on one row of every 128-row tile (plus the batch's first and
    last rows and the last row of every pair tile) within tolerance."""
    L = wl.make_layer_inputs(wl_name, layer=layer_idx)
    w = prep(L)
    x = x_dev(L.x_bits)
    y = wq.wq_linear_forward(w, x)
    codes, scales, g, xo, _ = wq.wq_quantize_activations(w, x)
    wq.wq_check_device_error(w)
    aq = oq(L)
    assert np.array_equal(g.cpu().numpy(), aq.g)
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    if L.omega.size:
        got, pad = side_out(xo, L.omega.size)
        assert np.array_equal(got, aq.x_omega) and not pad.any()
    rows = _tile_rows(L.M, 100 + layer_idx)
    ref = oracle.reference_forward(L, rows=rows)
    y_ref = ref[0]
    assert_y_close(L, y[torch.from_numpy(rows).cuda()], y_ref, rows, ref=ref)


@pytest.mark.parametrize("wide", ["1", "0"])
def test_full_size_long_k_both_gemm_schedules(wide, tuning):
    """The video-DiT down projection (M = 16384, K = 8960) on the CTA-pair schedule (its
    default) and on the single-CTA schedule, at full size, on sampled rows."""
    tuning("WQ_GEMM_WIDE", wide)
    L = wl.make_layer_inputs("video_dit", layer=3)
    w = prep(L)
    assert (wq.wq_gemm_schedule(w, L.M) == wq.WQ_GEMM_WIDE) == (wide == "1")   # K = 8960: one accumulator
    y = wq.wq_linear_forward(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    rows = _tile_rows(L.M, 300)
    ref = oracle.reference_forward(L, rows=rows)
    y_ref = ref[0]
    assert_y_close(L, y[torch.from_numpy(rows).cuda()], y_ref, rows, ref=ref)


# ------------------------------------------------------------------ batch-wide tensor scales
ACT_CASES = ["expert_small", "dit_r32_o64_ragged_n", "top2pct_o41_r24", "multi_tile_kstage_tail"]


@pytest.mark.parametrize("case", ACT_CASES)
@pytest.mark.parametrize("mode", ["tensor", "static"])
def test_batch_tensor_scale_modes(case, mode):
    """WQ_ACT_SCALE_TENSOR (one g from the whole batch's amax, two quantiser launches) and
    WQ_ACT_SCALE_STATIC (a calibrated g, one pass): codes, scales and g bit-exact against the
    oracle's per-tensor and fixed-g modes, x_Omega and U as in the per-row mode, y within
    tolerance of the oracle forward with that g."""
    L = layer(case)
    if mode == "static":
        # a calibrated g: the amax of a different batch of the same distribution, / 2688
        cal = wl.make_layer_inputs(CASES[case][0], **dict(CASES[case][1], M=64))
        ref = oracle.quantize_act(cal.x_bits, L.s, L.rotate, L.omega, per_tensor=True)
        g_cal = float(ref.g[0])
        w = wq.wq_prepare_weights(L.spec.K, L.spec.N, L.W, L.bias, L.s, L.L1, L.L2,
                                  L.omega if L.omega.size else None, rotate=L.rotate,
                                  act_scale=wq.WQ_ACT_SCALE_STATIC, act_gscale=g_cal)
        aq = oq(L, static_g=g_cal)
    else:
        w = wq.wq_prepare_weights(L.spec.K, L.spec.N, L.W, L.bias, L.s, L.L1, L.L2,
                                  L.omega if L.omega.size else None, rotate=L.rotate,
                                  act_scale=wq.WQ_ACT_SCALE_TENSOR)
        aq = oq(L, per_tensor=True)
    x = x_dev(L.x_bits)
    codes, scales, g, xo, u = wq.wq_quantize_activations(w, x)
    y = wq.wq_linear_forward(w, x)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w)
    assert np.all(g.cpu().numpy() == aq.g[0])
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    check_side(L, xo, u, aq)
    wqo = ow(L)
    U = oracle.lowrank_act(L.x_bits, wqo.P) if L.rank else None
    y_ref = oracle.linear_forward(aq, wqo, U, L.bias, per_tensor_act=True)
    assert_y_close(L, y, y_ref)


def test_side_strides_and_tuning_roundtrip():
    L = layer("top2pct_o41_r24")
    w = prep(L)
    assert wq.wq_side_strides(w) == (32, 64)
    old = wq.wq_get_tuning("WQ_GEMM_WIDE")
    wq.wq_set_tuning("WQ_GEMM_WIDE", 1)
    assert wq.wq_get_tuning("WQ_GEMM_WIDE") == 1
    wq.wq_set_tuning("WQ_GEMM_WIDE", old)
    with pytest.raises(wq.WqError):
        wq.wq_set_tuning("WQ_NO_SUCH_KNOB", 1)


# ------------------------------------------------------------------ W4A8 (A8-protected steps)
W4A8_CASES = ["expert_small", "dit_r32_o64_ragged_n", "top2pct_o41_r24", "multi_tile_kstage_tail",
              "rot_smooth_r32_o16", "min_k64_n16_m1"]


@pytest.mark.parametrize("case", W4A8_CASES)
@pytest.mark.parametrize("wide", ["0", "1"])
def test_w4a8_protected_step(case, wide, tuning):
    """QuantWAMs sec. 4.2 / sec. 5: a 4-bit layer at an A8-protected step.  e4m3 activation codes
    (read back as their bf16 values), row scales and fp16 kept channels bit-exact against the
    oracle; NVFP4 weight codes and scales bit-exact; y within tolerance on both GEMM schedules."""
    tuning("WQ_GEMM_WIDE", wide)
    L = layer(case)
    w = prep(L, mode=wq.WQ_MODE_W4A8)
    ex = wq.wq_export_weights(w)
    o = ow(L)
    assert np.array_equal(ex["codes"], o.codes) and np.array_equal(ex["scales"], o.scales)
    x = x_dev(L.x_bits)
    codes, _, g, xo, u = wq.wq_quantize_activations(w, x)
    y = wq.wq_linear_forward(w, x)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w)
    y_ref, aq, _, _ = oracle.reference_forward_w4a8(L)
    dec = torch.from_numpy(aq.q).view(torch.float8_e4m3fn).float().to(torch.bfloat16)
    assert torch.equal(codes.cpu().view(torch.int16), dec.view(torch.int16))
    assert np.array_equal(g.cpu().numpy(), aq.scale)
    if L.omega.size:
        got, pad = side_out(xo, L.omega.size)
        assert np.array_equal(got, aq.x_omega) and not pad.any()
    assert_y_close(L, y, y_ref)


# ------------------------------------------------------------------ Q-WAM projected complement
PROJ_CASES = ["tiny_full", "expert_small", "ragged_m130", "dit_r32_o64_ragged_n", "no_rotate_o16",
              "no_smooth_r64", "multi_tile_kstage_tail", "top2pct_o41_r24", "o5_r8", "o64_r40_no_rotate"]


def check_projected(L, w, x, rows=None, min_exact=0.9):
    """The projected-complement quantiser and forward against the oracle.  The projection takes
    u = bf16(x P) as an input; the GPU sums x P in fp32 and the oracle in fp64, so a row's u can
    differ by the bound of u_close.  On every row whose u is identical (at least min_exact of
    them) the codes, scales, g and x_Omega are bit-exact and y is within the y tolerance."""
    codes, scales, g, xo, u = wq.wq_quantize_activations(w, x, wq.WQ_SCALE_LAYOUT_ROWMAJOR)
    y = wq.wq_linear_forward(w, x)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w)
    y_ref, aq, o, U, _ = oracle.reference_forward_projected(L, rows=rows)
    sel = slice(None) if rows is None else torch.from_numpy(rows)
    xb = L.x_bits if rows is None else L.x_bits[rows]
    ug, pad = side_out(u[sel], L.rank)
    assert u_close(ug, U, xb, o.P).all() and not pad.any()
    same = (ug == U).all(axis=1)
    assert same.mean() >= min_exact, f"only {same.sum()} of {same.size} rows with identical u"
    idx = np.nonzero(same)[0]
    assert np.array_equal(g[sel].cpu().numpy()[idx], aq.g[idx])
    assert np.array_equal(scales[sel].cpu().numpy()[idx], aq.scales[idx])
    assert np.array_equal(codes[sel].cpu().numpy()[idx], aq.codes[idx])
    if L.omega.size:
        got, xpad = side_out(xo[sel], L.omega.size)
        assert np.array_equal(got[idx], aq.x_omega[idx]) and not xpad.any()
    r_idx = idx if rows is None else rows[idx]
    assert_y_close(L, y[torch.from_numpy(r_idx).cuda()], y_ref[idx], r_idx)


@pytest.mark.parametrize("case", PROJ_CASES)
def test_projected_complement(case):
    """Q-WAM abstract (Action-Subspace Protection): the activations' complement of the low-rank
    branch's subspace is what the quantiser sees.  Weights unchanged (bit-exact against the
    oracle's fold); the quantiser on the stream schedule (two launches)."""
    L = layer(case)
    w = prep(L, project=True)
    assert wq.wq_quant_schedule(w, L.M) == wq.WQ_QUANT_STREAM
    assert wq.wq_forward_path(w, L.M) == wq.WQ_PATH_TWO_KERNEL
    ex = wq.wq_export_weights(w)
    o = ow(L)
    assert np.array_equal(ex["codes"], o.codes) and np.array_equal(ex["scales"], o.scales)
    check_projected(L, w, x_dev(L.x_bits))


def test_projected_complement_changes_the_codes():
    """The projection is applied: the projected handle's codes differ from the plain handle's on
    the same input."""
    L = layer("dit_r32_o64_ragged_n")
    x = x_dev(L.x_bits)
    c0, *_ = wq.wq_quantize_activations(prep(L), x, wq.WQ_SCALE_LAYOUT_ROWMAJOR)
    c1, *_ = wq.wq_quantize_activations(prep(L, project=True), x, wq.WQ_SCALE_LAYOUT_ROWMAJOR)
    torch.cuda.synchronize()
    assert not torch.equal(c0, c1)


@pytest.mark.parametrize("wl_name", ["video_dit", "expert"])
def test_projected_complement_full_size(wl_name):
    """The full-size projection (video_dit's attention qkv input, the expert's up projection):
    one row of every 128-row tile plus the first and last rows."""
    L = wl.make_layer_inputs(wl_name, layer=0)
    w = prep(L, project=True)
    rows = _tile_rows(L.M, 31)
    check_projected(L, w, x_dev(L.x_bits), rows=rows, min_exact=0.85)


# ------------------------------------------------------------------ register-resident quantiser
@pytest.mark.parametrize("K,rank,n_omega", [(64, 16, 3), (192, 16, 5), (1088, 32, 64), (1536, 64, 16), (1536, 0, 0)])
def test_resident_quant_shapes(K, rank, n_omega, tuning):
    """The register-resident quantiser on its K range: one block, a pair and a lone block, 17 blocks
    (nine warps, the last with a lone block), twelve pairs with rank 64 (P read from L2) and twelve
    pairs without the branch; 72 rows (a ragged last tile).  Codes, scales, g and x_Omega
    bit-exact; U within its bound."""
    tuning("WQ_QUANT_SCHEDULE", "resident")
    L = wl.make_layer_inputs("video_dit", M=72, K=K, N=128, rank=rank, n_omega=n_omega)
    w = prep(L)
    assert wq.wq_quant_schedule(w, L.M) == wq.WQ_QUANT_RESIDENT
    x = x_dev(L.x_bits)
    codes, scales, g, xo, u = wq.wq_quantize_activations(w, x, wq.WQ_SCALE_LAYOUT_ROWMAJOR)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w)
    aq = oq(L)
    assert np.array_equal(g.cpu().numpy(), aq.g)
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    check_side(L, xo, u, aq)


# Kept channels in the patterns the copy-out has to get right: half a block's channels (all in
# the lower 32), a block with one channel at each end of both halves, the two blocks of one pair
# both with kept channels (a warp of the resident schedule, a cluster CTA's neighbouring warps),
# and most of the last block; 64 in all, sorted.
KEPT_PATTERN = np.array(sorted(list(range(128, 160)) + [192 + 31, 192 + 32, 192 + 63] + [256, 256 + 33] +
                               [320 + 5, 320 + 40, 320 + 62] + list(range(1472, 1496))), dtype=np.int32)


@pytest.mark.parametrize("schedule", ["cluster", "stream", "resident"])
def test_kept_channel_patterns(schedule, tuning):
    """x_Omega, codes, scales and g bit-exact and U within its bound for a hand-placed Omega
    (KEPT_PATTERN) on every quantiser schedule; 200 rows (a ragged last tile)."""
    import dataclasses
    tuning("WQ_QUANT_SCHEDULE", schedule)
    L = wl.make_layer_inputs("video_dit", M=200, K=1536, N=128, rank=32, n_omega=64)
    L = dataclasses.replace(L, omega=KEPT_PATTERN.copy())
    assert KEPT_PATTERN.size == 64 and np.all(np.diff(KEPT_PATTERN) > 0)
    w = prep(L)
    want = {"cluster": wq.WQ_QUANT_CLUSTER, "stream": wq.WQ_QUANT_STREAM, "resident": wq.WQ_QUANT_RESIDENT}[schedule]
    assert wq.wq_quant_schedule(w, L.M) == want
    x = x_dev(L.x_bits)
    codes, scales, g, xo, u = wq.wq_quantize_activations(w, x, wq.WQ_SCALE_LAYOUT_ROWMAJOR)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w)
    aq = oq(L)
    assert np.array_equal(g.cpu().numpy(), aq.g)
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    check_side(L, xo, u, aq)


@pytest.mark.parametrize("case", list(CASES))
def test_forward_parity_resident_quantiser(case, tuning):
    """The whole forward with the register-resident quantiser feeding the GEMM (a case whose K is
    wider than 1536 takes the stream schedule)."""
    tuning("WQ_QUANT_SCHEDULE", "resident")
    tuning("WQ_FUSED", "0")
    L = layer(case)
    w = prep(L)
    y = wq.wq_linear_forward(w, x_dev(L.x_bits))
    wq.wq_check_device_error(w)
    ref = oracle.reference_forward(L)
    y_ref = ref[0]
    assert_y_close(L, y, y_ref, ref=ref)


# ------------------------------------------------------------------ exhaustive value sweep
def _sweep_rows():
    """Rows of K = 1024 whose first 16-block is [2688, 0, ...] (so g = amax / 2688 = 1) and whose
    other 63 blocks each hold a maximum 6 dec(c) (so the block's e4m3 scale is exactly code c)
    and 15 values from every finite bf16 value v with |v| <= 6 dec(c), for every scale code
    c = 1 .. 126: each value meets each scale it can sit under."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = bits[(bits & 0x7F80) != 0x7F80]
    vals = wl.bf16_from_bits(finite).astype(np.float64)
    e = np.arange(1, 127)
    dec = np.where((e >> 3) == 0, (e & 7) * 2.0 ** -9, (1 + (e & 7) / 8) * 2.0 ** ((e >> 3) - 7))
    blocks = []
    for c, d in zip(e, dec):
        bm = 6.0 * d
        sel = finite[np.abs(vals) <= bm]
        pad = (-sel.size) % 15
        sel = np.concatenate([sel, np.zeros(pad, np.uint16)]).reshape(-1, 15)
        head = np.full((sel.shape[0], 1), wl.bf16_bits(np.array([bm], np.float32))[0], np.uint16)
        blocks.append(np.concatenate([head, sel], axis=1))
    blocks = np.concatenate(blocks)                        # [n, 16]
    nb = 63
    blocks = np.concatenate([blocks, np.zeros(((-len(blocks)) % nb, 16), np.uint16)])
    rows = blocks.reshape(-1, nb * 16)
    first = np.zeros((rows.shape[0], 16), np.uint16)
    first[:, 0] = wl.bf16_bits(np.array([2688.0], np.float32))[0]
    return np.ascontiguousarray(np.concatenate([first, rows], axis=1))


@pytest.mark.parametrize("schedule", ["stream", "cluster", "resident"])
def test_every_bf16_value_under_every_scale(schedule, tuning):
    """Every finite bf16 value quantised under every e4m3 block scale it can sit under (g = 1, no
    smoothing, no rotation, no branches), through wq_quantize_activations on each schedule:
    codes, scales and g bit-exact against the oracle."""
    tuning("WQ_QUANT_SCHEDULE", schedule)
    x_bits = _sweep_rows()
    M, K = x_bits.shape
    W = np.random.default_rng(11).standard_normal((K, 16)).astype(np.float32) * 0.02
    w = wq.wq_prepare_weights(K, 16, W, rotate=False)
    want = {"stream": wq.WQ_QUANT_STREAM, "cluster": wq.WQ_QUANT_CLUSTER, "resident": wq.WQ_QUANT_RESIDENT}[schedule]
    assert wq.wq_quant_schedule(w, M) == want
    codes, scales, g, _, _ = wq.wq_quantize_activations(w, x_dev(x_bits), wq.WQ_SCALE_LAYOUT_ROWMAJOR)
    torch.cuda.synchronize()
    wq.wq_check_device_error(w)
    aq = oracle.quantize_act(x_bits, None, False, None)
    assert np.all(aq.g == 1.0)
    assert np.array_equal(g.cpu().numpy(), aq.g)
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
