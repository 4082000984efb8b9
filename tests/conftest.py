import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkda")
    config.addinivalue_line("markers", "slow: larger CPU cases")


@pytest.fixture(scope="session")
def kda_gpu():
    """The CUDA binding on cuda:0; fails loudly when the library is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_kda_gb300 as kda
    kda.load()  # raises if libkda.so is absent
    return kda


def pytest_sessionfinish(session, exitstatus):
    """With KDA_PARITY_REPORT set, write the errors the parity tests measured
    per named workload (raw max-abs and excess over the half-ulp allowance)."""
    path = os.environ.get("KDA_PARITY_REPORT")
    if not path:
        return
    from kda_testutil import PARITY_ERRORS
    if PARITY_ERRORS:
        import json
        with open(path, "w") as f:
            json.dump(PARITY_ERRORS, f, indent=1, sort_keys=True)
