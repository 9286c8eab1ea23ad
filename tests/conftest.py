import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def synth_lib():
    import synth
    synth.build()
    return synth


# Routing near-tie counts and output errors of the full-size parity cases,
# printed at the end of the run (the tolerance statement asks for the tokens
# excluded as near ties to be counted and reported).
_PARITY_LINES = []


@pytest.fixture(scope="session")
def parity_report():
    def make(name):
        def report(rep, err, ref):
            _PARITY_LINES.append(
                f"{name}: tokens {rep.n_tokens}, near ties (k-th/(k+1)-th gap < 1e-5, "
                f"excluded) {rep.n_near_tie}, ties inside the top k (ids compared as sets) "
                f"{rep.n_inner_tie}, max|gpu-oracle| {err:.3e} = {err / ref:.2e} x max|oracle|")
        return report
    return make


def pytest_terminal_summary(terminalreporter):
    if _PARITY_LINES:
        terminalreporter.write_sep("-", "parity against the oracle (full-size workloads)")
        for line in _PARITY_LINES:
            terminalreporter.write_line(line)
