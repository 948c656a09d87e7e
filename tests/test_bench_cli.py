"""bench.py's command line on a machine without a GPU: the options parse, and
the reference arm prints its one JSON line with the reason it cannot run
instead of failing."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT, gpu_available


def run(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=300)


def test_help_lists_the_contract_options():
    r = run("--help")
    assert r.returncode == 0
    for opt in ("--gpus", "--steps", "--warmup", "--impl", "--workload"):
        assert opt in r.stdout


@pytest.mark.skipif(gpu_available(), reason="checks the behaviour without a GPU")
def test_reference_arm_without_gpu_reports_unavailable():
    r = run("--impl", "reference", "--steps", "1", "--warmup", "1")
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "unavailable" in line
