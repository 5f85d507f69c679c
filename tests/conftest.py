import os
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for _p in (ROOT, HERE):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree if needed; its calls need a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_151_gb300 import pa
    pa.load()
    return pa


def pytest_terminal_summary(terminalreporter):
    """Print the whole-output parity figures of the full-size workloads."""
    try:
        import fullsize
    except ImportError:
        return
    if not fullsize.RESULTS:
        return
    tr = terminalreporter
    tr.section("full-size parity against the fp64 oracle (every output element)")
    for name, n, err, rel, secs in fullsize.RESULTS:
        tr.write_line(f"{name:<48} {n:>10} elements  max|err| {err:.3e}  "
                      f"rel L2 {rel:.3e}  oracle {secs:6.1f} s")
