import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    # a planted oracle mistake (tests/oracle_mutations.py), only in the child
    # runs of tests/test_oracle_mutations.py
    name = os.environ.get("QMUON_PLANT_ORACLE_MISTAKE")
    if name:
        sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
        import oracle_mutations
        oracle_mutations.plant(name)


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
