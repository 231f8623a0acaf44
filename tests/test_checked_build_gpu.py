"""The bounds-checked build (-DZERO_CHECKED) over every kernel path.

compute-sanitizer is not used; instead the checked library tests each global
index against its buffer before the access and records the first failure (site, index) in
the status word without trapping. tests/checked_build_scenarios.py drives every kernel path
(misaligned fused all-gather stores, shards and per-bucket gathers, generic rank counts,
hybrid sharding, ZeRO-2 streaming, save / load across layouts, the allocation-free norm)
against it in a child process, compares each with the oracle and requires no failed check.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_reports_no_out_of_bounds_access():
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_build_scenarios.py")], capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "all scenarios clean" in r.stdout
