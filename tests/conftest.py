import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")



_KNOB_DEFAULTS = {"WQ_FUSED": 0, "WQ_GEMM_SPLIT": 0, "WQ_GEMM_WIDE": -1, "WQ_GEMM_PUSH": -1,
                  "WQ_GEMM_STAGES": 0, "WQ_QUANT_SCHEDULE": -1, "WQ_QUANT_SPLIT": 0,
                  "WQ_QUANT_CTAS_PER_SM": 0, "WQ_GEMM_DB": -1}


@pytest.fixture
def tuning():
    """Pin schedule knobs through wq_set_tuning for one test; every knob the test touched goes
    back to its automatic value afterwards."""
    import w4a4_nvfp4_quantized_wq_b300 as wq
    touched = []

    def set_knob(name, value):
        if isinstance(value, str):
            value = {"stream": 1, "cluster": 0, "resident": 2}.get(value, None) if not value.lstrip("-").isdigit() else int(value)
        wq.wq_set_tuning(name, int(value))
        touched.append(name)

    yield set_knob
    for name in touched:
        wq.wq_set_tuning(name, _KNOB_DEFAULTS[name])
