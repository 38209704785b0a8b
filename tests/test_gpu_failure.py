"""The failure path of the kernels' bounded waits, made to run out on purpose without a fault.

Every barrier wait in the library's kernels gives up after a time limit (2 s of global time),
records a site code in a device flag and releases the CTA's other waiters through an abort
flag; the host then reads WQ_ERR_TIMEOUT.  The self-test kernel waits on an mbarrier that
nothing arrives on -- no trap, no bad address, no endless loop -- and the test checks the
status, the recorded site, both waits' durations (the second waiter is released by the abort
flag before its own limit), and that a forward on the same context still matches the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import w4a4_nvfp4_quantized_wq_b300 as wq
import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_reports_and_leaves_the_context_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a4_nvfp4_quantized_wq_b300 import build
    build.build_library()
    torch.cuda.set_device(0)

    st, site, waited, released = wq.wq_selftest_wait_timeout()
    assert st == wq.WQ_ERR_TIMEOUT
    assert "site 91" in wq.wq_last_error()
    assert site == 91                       # the first wait's site; the released one records none
    assert released == 2
    assert 2000.0 <= waited[0] < 2400.0     # its own limit
    assert 2000.0 <= waited[1] < 2400.0     # counted from 0.5 s earlier: its own limit would be 2.5 s

    # the context is still usable: a forward afterwards matches the oracle
    L = wl.make_layer_inputs("tiny")
    w = wq.wq_prepare_weights(L.spec.K, L.spec.N, L.W, L.bias, L.s, L.L1, L.L2,
                              L.omega if L.omega.size else None, rotate=L.rotate)
    x = torch.from_numpy(np.ascontiguousarray(L.x_bits).view(np.int16)).view(torch.bfloat16).cuda()
    y = wq.wq_linear_forward(w, x)
    wq.wq_check_device_error(w)
    y_ref, *_ = oracle.reference_forward(L)
    xn = np.linalg.norm(L.x_f32.astype(np.float64), axis=1)[:, None]
    wn = np.linalg.norm(L.W.astype(np.float64), axis=0)[None, :]
    tol = 1e-3 * (np.abs(y_ref) + xn * wn / np.sqrt(L.spec.K)) + 2.0 ** -8 * np.abs(y_ref)
    assert (np.abs(y.float().cpu().numpy().astype(np.float64) - y_ref) <= tol).all()
