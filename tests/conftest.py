import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


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


def pytest_terminal_summary(terminalreporter):
    """Boundary swaps of the GPU parity cases (entries selected differently from the oracle
    where the oracle scores tie the k-th score within the score tolerance), also written to
    $INDEXER_SWAPS_JSON, or to gpurun_out/boundary_swaps.json when that folder exists."""
    try:
        from tests import cases as C
    except Exception:  # pragma: no cover
        return
    if not C.SWAPS:
        return
    import json
    terminalreporter.section("boundary swaps (selected entries that differ from the oracle at the k-th score)")
    for case, v in sorted(C.SWAPS.items()):
        terminalreporter.write_line(f"{case}: {v['swaps']} swaps in {v['selected']} selected entries "
                                    f"({v['rows']} rows)")
    path = os.environ.get("INDEXER_SWAPS_JSON")
    if not path and os.path.isdir(os.path.join(ROOT, "gpurun_out")):
        path = os.path.join(ROOT, "gpurun_out", "boundary_swaps.json")
    if path:
        with open(path, "w") as f:
            json.dump(C.SWAPS, f, indent=1, sort_keys=True)
