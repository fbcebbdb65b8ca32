import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle():
    from oracle import oracle as O
    O.build()
    return O


def pytest_terminal_summary(terminalreporter):
    """Counts of GPU tokens that differ from the oracle's (allowed near ties and
    bf16-boundary cases), per checked workload."""
    try:
        from parity import REPORT
    except ImportError:
        return
    if not REPORT:
        return
    terminalreporter.write_line("parity counts (steps: same / near-tie / bf16-boundary; max |logit error|):")
    for label, st in sorted(REPORT.items()):
        terminalreporter.write_line(f"  {label}: {st.steps}: {st.same} / {st.near_tie} / {st.bf16_boundary}; "
                                    f"{st.max_abs_err:.3g}")
