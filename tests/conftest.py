import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


def pytest_collection_modifyitems(config, items):
    # the no-allocation entry point's test file sorts last by name; keep the
    # rest in file order
    items.sort(key=lambda it: 1 if os.path.basename(str(it.fspath)).startswith("test_zz") else 0)


@pytest.fixture(scope="session")
def gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_quantized_kv_store_gb300 as kvq
    kvq.load()  # raises if the extension is missing
    return kvq
