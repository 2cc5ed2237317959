import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def tune():
    """Sets a library tuning switch (dh_set_tuning) for one test and restores the default after it."""
    from speculative_decoding_draft_dh_gb300 import binding as dh
    changed = []

    def set_switch(name, value):
        dh.set_tuning(name, value)
        changed.append(name)

    yield set_switch
    for name in changed:
        dh.set_tuning(name, None)
