import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


import pytest


@pytest.fixture
def tune():
    """Set the library's planner overrides (q8_set_tuning) for one test; the previous values come back afterwards.
    tune(ksplit=4), tune(gemm=0 or 1), tune(norm_fold=1) -- see include/q8_gemv.h, Q8_TUNE_*."""
    import q8_block_quantized_gemv_gb300 as q8
    saved = {}

    def set_(**overrides):
        for k, v in overrides.items():
            saved.setdefault(k, q8.get_tuning(k))
            q8.set_tuning(k, v)

    yield set_
    for k, v in saved.items():
        q8.set_tuning(k, v)
