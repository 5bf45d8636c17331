import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libsbt.so")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def sbt_ctx():
    """One library context on cuda:0 (the build must exist: no fallback)."""
    import scatter_boundary_tile_gb300 as sbt

    sbt.load_library()
    ctx = sbt.Context(0)
    yield ctx
    ctx.close()


@pytest.fixture
def ctx(sbt_ctx):
    sbt_ctx.set_path("auto")
    yield sbt_ctx
    sbt_ctx.set_path("auto")
    sbt_ctx.check_status()
