"""The bounds-checking build (-DHALO_DEBUG): every slot index a kernel gathers
from or scatters to is checked before use, and a bad one is reported as
HALO_EBOUNDS instead of being accessed.  On correct plans it must report
nothing and give the same bits as the release build (the checks stand in for
a memory sanitizer, which this pool does not offer)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_reports_no_bad_index_and_matches_the_oracle():
    from domain_decomposition_halo_build_gb300 import _build
    lib = _build.build(debug=True)
    env = dict(os.environ, HALO_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_parity_run.py")],
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build ok" in r.stdout
