"""Shared pytest setup: the ``gpu`` marker and repository import path."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    """GPU tests fail loudly (not skip) when selected without a GPU: a silent
    skip would read as a pass."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(pytest.mark.skipif(
                os.environ.get("PKV_REQUIRE_GPU") != "1",
                reason="no CUDA device"))
