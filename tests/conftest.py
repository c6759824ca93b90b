import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    gu = sys.modules.get("tests.gpu_util")
    use = getattr(gu, "ULP_ALLOWANCE_USE", None) if gu else None
    if use and use["compared"]:
        terminalreporter.write_line(
            f"prefill tolerance: {use['needed']} of {use['compared']} compared elements were "
            f"above 1e-2 and passed through the one-ulp allowance")
