import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_sessionfinish(session, exitstatus):
    """Flips (near-tie token or acceptance differences between the CUDA path and
    the oracle) summed over the session must stay below 0.1 % of the compared
    tokens (checked once at least 1000 tokens were compared; smaller runs are
    held to the per-comparison rule alone)."""
    import parity
    led = parity.LEDGER
    if led["compared"] >= 1000 and led["flips"] >= 0.001 * led["compared"]:
        session.exitstatus = pytest.ExitCode.TESTS_FAILED
        print(f"\nparity: {led['flips']} flips in {led['compared']} compared tokens, not below 0.1 %")


def pytest_terminal_summary(terminalreporter):
    import parity
    led = parity.LEDGER
    if led["compared"]:
        terminalreporter.write_line(
            f"parity ledger: {led['flips']} flips in {led['compared']} compared tokens over "
            f"{led['comparisons']} comparisons ({100.0 * led['flips'] / led['compared']:.4f} %)")
