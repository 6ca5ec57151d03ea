"""Shared test configuration.

``-m "not gpu"`` runs the CPU suite: the oracle against its pins, the host
helpers and the C-ABI library's exports and argument checks.  ``-m gpu``
runs the parity tests that call the CUDA library through its C ABI.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Rows of whitespace-separated fields; '#' starts a comment."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def oracle_lib():
    from oracle import kq_oracle
    kq_oracle.lib()
    return kq_oracle


def build_c_helper(tmpdir, name):
    """Compile tests/<name>.c into a shared object under tmpdir."""
    src = os.path.join(HERE, name + ".c")
    out = os.path.join(str(tmpdir), "lib" + name + ".so")
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    "-std=c11", "-o", out, src, "-lm"], check=True)
    return out
