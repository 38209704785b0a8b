"""GPU parity of the VAE Conv3d implicit GEMM against the direct-convolution oracle.

Bar: input voxel codes, scales and the tensor scale bit-exact; weight codes/scales bit-exact;
y within 1e-3 (|y| + ||a_row|| ||w_col|| / sqrt(K)) + 2^-8 |y|, with a_row the row of the
implicit GEMM (the 27 voxels a tap reaches, zero in the padding).
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


def run_case(T, H, W, C_in, C_out, vox=None, B=1):
    xb, w = wl.make_conv_inputs(T=T, H=H, W=W, C_in=C_in, C_out=C_out, B=B)
    V1 = T * H * W
    hw = wq.wq_prepare_conv3d(w)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    y = wq.wq_conv3d_forward(hw, x)
    codes, scales, g = wq.wq_quantize_conv3d_input(hw, x)
    wq.wq_check_device_error(hw)
    if vox is None:
        vox = np.arange(B * V1)
    y_ref, aq, wqo = oracle.conv3d_reference(xb, w, vox)
    assert np.float32(g.item()) == aq.g[0]
    assert np.array_equal(scales.cpu().numpy(), aq.scales)
    assert np.array_equal(codes.cpu().numpy(), aq.codes)
    ex = wq.wq_export_weights(hw)
    assert np.array_equal(ex["codes"], wqo.codes) and np.array_equal(ex["scales"], wqo.scales)
    # tolerance from the implicit-GEMM rows of the original input
    xf = wl.bf16_from_bits(xb).astype(np.float64)                    # [B, C, T, H, W]
    xp = np.zeros((B, C_in, T + 2, H + 2, W + 2))
    xp[:, :, 1:-1, 1:-1, 1:-1] = xf
    b, lv = vox // V1, vox % V1
    d, h, ww = lv // (H * W), (lv // W) % H, lv % W
    an = np.sqrt(sum((xp[b, :, d + kd, h + kh, ww + kw] ** 2).sum(axis=1)
                     for kd in range(3) for kh in range(3) for kw in range(3)))
    wn = np.linalg.norm(oracle.conv_weight_matrix(w).astype(np.float64), axis=0)
    tol = 1e-3 * (np.abs(y_ref) + an[:, None] * wn[None, :] / np.sqrt(27 * C_in)) + 2.0 ** -8 * np.abs(y_ref)
    yall = y.reshape(B, C_out, V1).float().cpu().numpy().astype(np.float64)
    yg = yall[b, :, lv]
    err = np.abs(yg - y_ref)
    assert (err <= tol).all(), f"{(err > tol).sum()} of {err.size} outside tolerance, worst {np.max(err - tol):.3g}"


def test_conv3d_small_all_voxels():
    run_case(3, 5, 8, 128, 32)


def test_conv3d_several_tiles_partial_n():
    run_case(2, 7, 24, 256, 48)


def test_conv3d_two_column_tiles_partial():
    """A work item with two column tiles, the second partial (C_out = 160)."""
    run_case(2, 6, 16, 128, 160)


def test_conv3d_column_groups_of_three_and_one():
    """C_out = 512: four column tiles, split into a work item of three and one of one."""
    run_case(2, 6, 16, 128, 512)


def test_conv3d_batch_of_two_all_voxels():
    """Batch 2 (320 voxels per sample, so 128-voxel tiles straddle the two samples): one tensor
    scale over the batch, and no tap reaches from one sample into the other."""
    run_case(4, 5, 16, 128, 48, B=2)


def test_conv3d_batch_of_three_odd_volume():
    run_case(3, 3, 8, 256, 32, B=3)


def test_conv3d_rejects_other_kernels():
    w = np.zeros((16, 128, 1, 3, 3), np.float32)
    with pytest.raises(wq.WqError) as e:
        wq.wq_prepare_conv3d(w)
    assert e.value.status == wq.WQ_ERR_UNSUPPORTED
    with pytest.raises(wq.WqError) as e:
        wq.wq_prepare_conv3d(np.zeros((16, 128, 3, 3, 3), np.float32), pad=0)
    assert e.value.status == wq.WQ_ERR_UNSUPPORTED


def test_conv3d_vae_full_size_every_work_item_and_face():
    """The full VAE convolution: one voxel in every 128-voxel work item of the GEMM, the volume's
    corners, and voxels on all six padding faces."""
    T, H, W = 5, 60, 104
    V = T * H * W
    rng = np.random.default_rng(9)
    vox = {0, V - 1}
    for t in range(0, V, 128):
        vox.add(t + int(rng.integers(0, min(128, V - t))))
    for _ in range(6):
        d, h, w_ = int(rng.integers(0, T)), int(rng.integers(0, H)), int(rng.integers(0, W))
        for dd, hh, ww_ in ((0, h, w_), (T - 1, h, w_), (d, 0, w_), (d, H - 1, w_), (d, h, 0), (d, h, W - 1)):
            vox.add((dd * H + hh) * W + ww_)
    for c in [W - 1, (H - 1) * W, H * W - 1, (T - 1) * H * W]:
        vox.add(c)
    run_case(T, H, W, 384, 384, np.array(sorted(vox)))
