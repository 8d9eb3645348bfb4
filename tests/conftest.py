import multiprocessing
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    """GPU tests are skipped, not failed, on a machine without a GPU, unless
    they were asked for explicitly with ``-m gpu``."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    markexpr = config.getoption("-m") or ""
    if markexpr.strip() == "gpu":
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def parity_log(request):
    """(workload, excused exceptions, elements) of every whole-workload parity
    check, printed at the end of the run."""
    log = []
    request.config._fp4q_parity_log = log
    return log


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    log = getattr(config, "_fp4q_parity_log", None)
    if not log:
        return
    terminalreporter.write_sep("-", "whole-workload parity: every row against the oracle")
    for name, exc, n in log:
        terminalreporter.write_line(f"{name}: {exc} excused boundary exceptions in {n} elements "
                                    f"({exc / max(n, 1):.2e}; bound 1e-4)")


@pytest.fixture(scope="session")
def oracle_pool():
    """Oracle workers for full-size parity: spawned (never forked after CUDA
    is initialised), one per host core, single-threaded numpy each."""
    n = max(1, min(32, len(os.sched_getaffinity(0))))
    keep = os.environ.get("OMP_NUM_THREADS")
    os.environ["OMP_NUM_THREADS"] = "1"
    try:
        p = multiprocessing.get_context("spawn").Pool(n)
    finally:
        if keep is None:
            os.environ.pop("OMP_NUM_THREADS", None)
        else:
            os.environ["OMP_NUM_THREADS"] = keep
    yield p
    p.close()
    p.join()
