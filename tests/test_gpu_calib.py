"""GPU parity of the on-device outlier calibration (QuantWAMs sec. 3.1 Eq. (1)-(3), one context)
against the oracle: z(c) within 1e-12 relative (fp64 sums in another order of the same exact
squares) and the Top-K set equal to the oracle's, except where the oracle's z at the boundary
differ by less than that tolerance (then either choice is correct)."""
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


def check_topk(om_gpu, z_ref, n):
    om_ref = oracle.topk_channels(z_ref, n)
    if np.array_equal(om_gpu, om_ref):
        return
    boundary = np.sort(z_ref)[::-1][n - 1]
    diff = set(om_gpu.tolist()) ^ set(om_ref.tolist())
    assert all(abs(z_ref[c] - boundary) <= 1e-12 * boundary for c in diff), sorted(diff)
    assert np.all(np.diff(om_gpu) > 0) and om_gpu.size == n


@pytest.mark.parametrize("kw,after,n", [(dict(M=300, K=512), False, 16), (dict(M=1500, K=1024), True, 41),
                                        (dict(M=1, K=64), False, 3), (dict(M=2049, K=256, smooth=False), False, 0)])
def test_pooled_energy_and_topk(kw, after, n):
    L = wl.make_layer_inputs("video_dit", N=16, rank=0, n_omega=0, smooth_after=after, **kw)
    x = torch.from_numpy(L.x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    z, om = wq.wq_calibrate_outliers(x, L.s, True, int(after), n)
    torch.cuda.synchronize()
    z_ref = oracle.pooled_energy(L.x_bits, L.s, True, after)
    np.testing.assert_allclose(z.cpu().numpy(), z_ref, rtol=1e-12, atol=0)
    if n:
        check_topk(om.cpu().numpy(), z_ref, n)


def test_calibration_full_size_video_dit_down():
    """The video-DiT down projection's input (M = 16384, K = 8960): z of every channel and the
    top 64, as the workload's Omega is chosen."""
    L = wl.make_layer_inputs("video_dit", layer=3, N=16, rank=0, n_omega=0)
    x = torch.from_numpy(L.x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    z, om = wq.wq_calibrate_outliers(x, L.s, True, 0, 64)
    torch.cuda.synchronize()
    z_ref = oracle.pooled_energy(L.x_bits, L.s, True)
    np.testing.assert_allclose(z.cpu().numpy(), z_ref, rtol=1e-12, atol=0)
    check_topk(om.cpu().numpy(), z_ref, 64)


def test_calibration_ties_go_to_the_lower_index():
    """Rows with several channels of identical energy: the selection follows the index rule."""
    K = 128
    x = np.zeros((8, K), np.float32)
    x[:, [5, 9, 70, 100]] = 2.0
    x[:, 40] = 3.0
    bits = wl.bf16_bits(x)
    xd = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    z, om = wq.wq_calibrate_outliers(xd, None, False, 0, 3)
    torch.cuda.synchronize()
    assert om.cpu().tolist() == [5, 9, 40]
    np.testing.assert_array_equal(z.cpu().numpy(), oracle.pooled_energy(bits, None, False))
