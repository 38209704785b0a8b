"""The synthetic inputs every parity test and bench line uses are seeded: the same request
gives the same bits, different layers and workloads give different draws, and the planted
structure (outlier channels, Omega, low-rank factors) has the stated shapes.  No GPU."""
import numpy as np
import pytest

import workloads as wl


def _arrays(L):
    out = {"x": L.x_bits, "W": L.W}
    for k in ("bias", "s", "L1", "L2", "omega"):
        v = getattr(L, k, None)
        if v is not None:
            out[k] = v
    return out


@pytest.mark.parametrize("name,kw", [("expert", dict(M=20, K=256, N=128)),
                                     ("video_dit", dict(M=24, K=512, N=96, rank=32, n_omega=16)),
                                     ("backbone", dict(layer=1, M=9, K=256, N=64))])
def test_same_request_same_bits(name, kw):
    a, b = _arrays(wl.make_layer_inputs(name, **kw)), _arrays(wl.make_layer_inputs(name, **kw))
    assert a.keys() == b.keys()
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_layers_and_workloads_draw_differently():
    e0 = wl.make_layer_inputs("expert", layer=0, M=8, K=256, N=64)
    e1 = wl.make_layer_inputs("expert", layer=1, M=8, K=256, N=64)
    v0 = wl.make_layer_inputs("video_dit", layer=0, M=8, K=256, N=64)
    assert not np.array_equal(e0.x_bits, e1.x_bits) and not np.array_equal(e0.W, e1.W)
    assert not np.array_equal(e0.W, v0.W)


def test_shapes_and_planted_structure():
    L = wl.make_layer_inputs("video_dit", M=32, K=512, N=96, rank=32, n_omega=16)
    assert L.x_bits.shape == (32, 512) and L.x_bits.dtype == np.uint16
    assert L.W.shape == (512, 96)
    assert L.L1.shape[1] == 32 and L.L2.shape[0] == 32
    om = L.omega
    assert om.size == 16 and np.all(np.diff(om) > 0) and om.min() >= 0 and om.max() < 512
    ch = wl.outlier_channels(256, 4)
    assert list(ch) == [32, 96, 160, 224]          # floor((i + 1/2) K / n)


def test_conv_inputs_are_seeded():
    a = wl.make_conv_inputs(T=2, H=4, W=8, C_in=128, C_out=32)
    b = wl.make_conv_inputs(T=2, H=4, W=8, C_in=128, C_out=32)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert a[0].shape[-4:] == (128, 2, 4, 8) and a[1].shape == (32, 128, 3, 3, 3)
