"""The bench's algorithmic byte counts (the numerators of every roofline fraction) against the
sizes of the arrays the operation actually reads and writes, taken from the oracle's outputs
on small layers.  No GPU is touched."""
import os
import sys

import numpy as np
import pytest

import oracle
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("kw", [dict(M=40, K=512, N=272, rank=32, n_omega=64),
                                dict(M=17, K=256, N=128, rank=16, n_omega=0),
                                dict(M=9, K=192, N=64, rank=0, n_omega=16, smooth=False)])
def test_w4a4_byte_counts_match_the_arrays(kw):
    L = wl.make_layer_inputs("video_dit", **kw)
    o = oracle.prepare_weights(L.W, L.s, L.L1, L.L2, L.omega, L.rotate)
    aq = oracle.quantize_act(L.x_bits, L.s, L.rotate, L.omega)
    r, n_out, smooth = L.rank, L.omega.size, L.s is not None
    U = oracle.lowrank_act(L.x_bits, o.P) if r else np.zeros((L.M, 0), np.uint16)
    x_omega = aq.x_omega if n_out else np.zeros((L.M, 0), np.uint16)
    W_omega = o.W_omega if n_out else np.zeros((0, L.spec.N), np.uint16)
    # quantiser: x in; codes, scales, row scales, U and x_O out (the per-layer constants P and
    # inv_s are not counted)
    q_bytes = L.x_bits.nbytes + aq.codes.nbytes + aq.scales.nbytes + aq.g.nbytes + U.nbytes + x_omega.nbytes
    assert bench.quant_algorithmic_bytes(L.M, L.spec.K, r, n_out, smooth) == q_bytes
    # GEMM: both operands with their scales, the row scales, the side operands, bias, y out
    y_bytes = L.M * L.spec.N * 2
    g_bytes = aq.codes.nbytes + aq.scales.nbytes + aq.g.nbytes + o.codes.nbytes + o.scales.nbytes + \
        o.Q.nbytes * (r > 0) + W_omega.nbytes + U.nbytes + x_omega.nbytes + \
        (L.bias.nbytes if L.bias is not None else 0) + y_bytes
    assert bench.gemm_algorithmic_bytes(L.M, L.spec.K, L.spec.N, r, n_out, L.bias is not None) == g_bytes


def test_w8a8_byte_counts_match_the_arrays():
    L = wl.make_layer_inputs("backbone", layer=1, M=33, K=512, N=96)
    w8 = oracle.prepare_weights_int8(L.W, L.s, L.rotate)
    a8 = oracle.quantize_act_int8(L.x_bits, L.s, L.rotate)
    inv_s = np.zeros(L.spec.K, np.float32)
    assert bench.quant8_algorithmic_bytes(L.M, L.spec.K, True) == \
        L.x_bits.nbytes + inv_s.nbytes + a8.q.nbytes + a8.scale.nbytes
    assert bench.gemm8_algorithmic_bytes(L.M, L.spec.K, L.spec.N, True) == \
        a8.q.nbytes + a8.scale.nbytes + w8.q.nbytes + w8.scale.nbytes + L.bias.nbytes + L.M * L.spec.N * 2


def test_traffic_figure_is_used_only_for_the_code_it_measured(tmp_path, monkeypatch):
    """A stored ncu traffic figure is reported only while the kernel sources hash to the value
    recorded with it."""
    import json
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.kernel_source_hash()
    (prof / "traffic.json").write_text(json.dumps({"w": {"k": {"dram_bytes_per_launch": 123.0, "source_hash": h},
                                                         "old": {"dram_bytes_per_launch": 7.0, "source_hash": "x"}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: h)
    assert bench.profiled_traffic("k", "w") == 123.0
    assert bench.profiled_traffic("old", "w") is None
    assert bench.profiled_traffic("missing", "w") is None


def test_kernel_roofline_picks_the_binding_term():
    """Roofline time of a launch = max(flops / P_fp4, bytes / HBM), P_fp4 = 6 x measured bf16."""
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}
    assert bench.fp4_peak_tflops(peaks) == 600.0
    r = bench.kernel_roofline(6e11, 1e6, 2.0, peaks)            # 1 ms of tensor time, 1 us of HBM time
    assert r["bound"] == "tensor" and abs(r["roofline_us"] - 1000.0) < 1e-9 and abs(r["frac"] - 0.5) < 1e-12
    r = bench.kernel_roofline(6e8, 1e9, 4.0, peaks)             # 1 us of tensor time, 1 ms of HBM time
    assert r["bound"] == "hbm" and abs(r["roofline_us"] - 1000.0) < 1e-9 and abs(r["frac"] - 0.25) < 1e-12
    r = bench.kernel_roofline(0.0, 2e6, 1.0, peaks)
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.002) < 1e-12


def test_default_workload_is_the_largest_config():
    import sys as _s
    argv = _s.argv
    try:
        _s.argv = ["bench.py"]
        a = bench.parse_args()
    finally:
        _s.argv = argv
    assert a.workload == "video_dit" and a.warmup >= 3 and a.steps >= 1
