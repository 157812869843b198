"""The exchange-checking build (-DRNN_CHECKS): every buffer the persistent
steps exchange through is poisoned before each launch and every slice that
lands in a CTA's shared memory is scanned for the poison, so a read before
the producers' write ends the call with RNN_INTERNAL.  Runs tests/checks_run.py
(its own process: the checking library is a second build) on K splits over
clusters and through global memory, batch parts, lengths, two layers and both
directions, GRU reset-before's two exchanges; every case must finish clean and
match the oracle, and an initial state holding the poison pattern (what a
slice read before its write looks like) must be reported."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checking_build_finds_no_early_read():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checks_run.py")], capture_output=True, text=True,
                       cwd=ROOT, timeout=1200)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "all checked" in r.stdout
    assert r.stdout.count("checked:") == 5
    # negative control: a poison-pattern value in the initial state is reported
    assert "checker fired on the poison pattern" in r.stdout
