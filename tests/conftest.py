import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library through its Python binding; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import megatron_tensor_block_gb300 as tb
    tb.load()
    return tb


def pytest_terminal_summary(terminalreporter):
    """Normwise and element-wise relative errors of every parity comparison
    made through ``tests/_parity.py`` in this session."""
    try:
        from tests import _parity
    except ImportError:
        return
    if not _parity.RECORDS:
        return
    tr = terminalreporter
    tr.section("parity: normwise | element-wise relative error")
    for test, what, n, e in _parity.RECORDS:
        tr.write_line(f"{n:9.2e} | {e:9.2e}  {test}{' ' + what if what else ''}")
