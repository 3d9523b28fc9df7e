"""Test configuration: the ``gpu`` marker and session-wide fixtures.

``-m "not gpu"`` runs on a CPU-only machine: the oracle against its pins, the
input generator, the host-side argument checks of the C-ABI library and the
multi-rank host logic.  ``-m gpu`` runs the CUDA parity tests through the
C-ABI on one GPU.
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and runs the CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def pa_lib_path():
    """Build libpa.so (if stale) through the entry point's builder and return its path."""
    import __graft_entry__
    return __graft_entry__._builder().build()


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True


def pytest_sessionfinish(session, exitstatus):
    """With PA_PARITY_LOG set, write every attention comparison's max-abs / mean-abs."""
    path = os.environ.get("PA_PARITY_LOG")
    mod = sys.modules.get("paged_steps")
    if not path or mod is None or not mod.RECORDS:
        return
    with open(path, "w") as f:
        json.dump(mod.RECORDS, f, indent=0)
