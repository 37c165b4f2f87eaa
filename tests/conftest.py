import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--mtp-library", default=None,
                     help="load this build of the library (e.g. the MTP_DEBUG build) in the GPU tests")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    from tests import gpu_util_paths

    gpu_util_paths.LIBRARY = config.getoption("--mtp-library")


def pytest_sessionfinish(session, exitstatus):
    # with --mtp-library, name the library builds this process mapped (the
    # debug-build test checks that the child ran on the build it asked for)
    if session.config.getoption("--mtp-library") and os.path.exists("/proc/self/maps"):
        libs = sorted({line.split()[-1] for line in open("/proc/self/maps") if "libmtprs" in line})
        print("\nmapped library builds: " + " ".join(os.path.basename(p) for p in libs))


def pytest_collection_modifyitems(config, items):
    # Tests marked gpu are skipped with a clear reason when no GPU is present,
    # so `-m "not gpu"` and a plain run both work on CPU-only machines.
    try:
        import torch

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
