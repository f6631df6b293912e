import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


# Mismatch counts of the one-ulp parity checks (LayerNorm y, QKV-epilogue q and k: elements
# that differ from the oracle by one bf16 ulp), reported at the end of the run.
PARITY_COUNTS = []


def pytest_terminal_summary(terminalreporter):
    if not PARITY_COUNTS:
        return
    total = sum(n for _, n, _ in PARITY_COUNTS)
    elems = sum(e for _, _, e in PARITY_COUNTS)
    terminalreporter.write_line(
        f"one-ulp parity (LayerNorm y, QKV q/k): {len(PARITY_COUNTS)} checks, {elems} elements, "
        f"{total} differ from the oracle by 1 bf16 ulp (none by more)")
    for what, n, e in PARITY_COUNTS:
        if n:
            terminalreporter.write_line(f"  {what}: {n} of {e}")
