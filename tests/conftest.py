import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The largest bf16 ulp distance each sum check saw against the oracle."""
    mod = sys.modules.get("tests.test_parity_gpu")
    seen = getattr(mod, "MAX_ULP_SEEN", None) if mod is not None else None
    if seen:
        terminalreporter.write_line("max bf16 ulp vs the oracle: " + ", ".join(
            "%s %d" % (k, v) for k, v in sorted(seen.items())))
