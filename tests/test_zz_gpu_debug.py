"""The MTP_DEBUG build against the oracle: the device primitives of that
build check every shared-memory vector load, bulk copy, DSMEM address and
TMEM column they touch, and print a line starting with "MTP_DEBUG" for any
that fails (no trap; the access is skipped).  The whole GPU parity suite
runs in a child pytest on that build: it must pass and print no such
line."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_debug_build_parity_and_bounds():
    from mtp_speculative_decoding_row_gb300 import build as mtp_build

    lib = mtp_build.build(debug=True)
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-q", "-s", "-m",
           "gpu", "-p", "no:cacheprovider", "--mtp-library", lib]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=3000)
    out = r.stdout + r.stderr
    hits = [line for line in out.splitlines() if line.startswith("MTP_DEBUG")]
    assert not hits, "debug checks failed:\n" + "\n".join(hits[:20])
    assert r.returncode == 0, out[-4000:]
    assert " passed" in out, out[-2000:]
    mapped = [line for line in out.splitlines() if line.startswith("mapped library builds:")]
    assert mapped and "libmtprs_debug.so" in mapped[-1] and "libmtprs.so" not in mapped[-1].split(), mapped
