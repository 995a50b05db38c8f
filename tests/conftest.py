import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle():
    """The CPU oracle package.  PKV_ORACLE_DIR may point at another copy of
    it (the mutation test plants mistakes in such a copy)."""
    alt = os.environ.get("PKV_ORACLE_DIR")
    if alt:
        import importlib.util
        spec = importlib.util.spec_from_file_location(
            "oracle_under_test", os.path.join(alt, "__init__.py"),
            submodule_search_locations=[alt])
        O = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(O)
    else:
        import oracle as O
    O.build()
    return O


def _cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
