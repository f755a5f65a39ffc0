"""GPU runs of the bounds-checking build (LA_CHECK_BOUNDS): small parity cases
through every index path of the tensor-core kernels (ragged tails, packed and
empty sequences, both directions, key widths 64-256 and value tiles, grouped
heads, the sequence split, the gated form) with the checks compiled in, in a
process of its own that loads liblagb300_checked.so (tests/bounds_cases.py).
A failed check would come back from la_get_device_error as LA_ERR_BOUNDS
with its site; none may, and every checked case must match the oracle."""
import os
import subprocess
import sys

import pytest

from linear_attention_head_gb300 import build as libbuild

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounds_checked_build_runs_clean_and_matches_the_oracle():
    path = libbuild.build(checked=True)
    env = dict(os.environ, LA_LIBRARY=path)
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "bounds-checked cases ok" in r.stdout
