import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)



def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); parity of the CUDA path against the oracle")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # (case, relative L2, max abs / max |oracle|) of every layer-output parity
    # check, printed at the end of the run so that the margins show in quiet runs
    from tests.helpers import PARITY_REPORT
    if not PARITY_REPORT:
        return
    terminalreporter.section("layer-output parity against the oracle (bar: rel L2 <= 1e-3, max abs <= 1e-2 max|y|)")
    for case, rel, mx in PARITY_REPORT:
        terminalreporter.write_line(f"{case:70s} rel L2 {rel:.3e}   max abs / max|y| {mx:.3e}")
