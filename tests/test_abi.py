"""The C-ABI library builds, loads and exports every declared symbol; host
validation answers without touching a GPU (CPU-only tests)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import mtp_speculative_decoding_row_gb300 as mtp
from mtp_speculative_decoding_row_gb300 import build as mtp_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mtp_build.build()
    return mtp.load_library()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(?:int|const char \*|void)\s*\**\s*(mtp_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert {"mtp_rs_verify", "mtp_row_stats", "mtp_tv_loss_fwd_bwd", "mtp_status_string"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", mtp_build.LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = declared - exported
    assert not missing, missing
    for name in declared:
        assert hasattr(lib, name)


def test_status_strings(lib):
    assert mtp.mtp_status_string(0) == "ok"
    for s in range(1, 6):
        assert mtp.mtp_status_string(s) not in ("ok", "unknown status")


def test_host_validation_without_gpu(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)  # aligned, never dereferenced: validation fails first
    odd = P((1 << 20) + 8)
    # unsupported dtype
    assert lib.mtp_rs_verify(fake, fake, 7, fake, fake, fake, 4, 3, 10, fake, fake, None, None, None, None) == 2
    # bad gamma / V / B
    assert lib.mtp_rs_verify(fake, fake, 0, fake, fake, fake, 4, 0, 10, fake, fake, None, None, None, None) == 1
    assert lib.mtp_rs_verify(fake, fake, 0, fake, fake, fake, 4, 33, 10, fake, fake, None, None, None, None) == 1
    assert lib.mtp_rs_verify(fake, fake, 0, fake, fake, fake, 4, 3, 0, fake, fake, None, None, None, None) == 1
    assert lib.mtp_rs_verify(fake, fake, 0, fake, fake, fake, -1, 3, 10, fake, fake, None, None, None, None) == 1
    # B = 0 is a no-op
    assert lib.mtp_rs_verify(None, None, 0, None, None, None, 0, 3, 10, None, None, None, None, None, None) == 0
    # required pointers
    assert lib.mtp_rs_verify(fake, fake, 0, None, fake, fake, 4, 3, 10, fake, fake, None, None, None, None) == 1
    assert lib.mtp_rs_verify(fake, fake, 0, fake, fake, fake, 4, 3, 10, fake, fake, fake, None, None, None) == 1
    # misaligned logits
    assert lib.mtp_rs_verify(odd, fake, 0, fake, fake, fake, 4, 3, 10, fake, fake, None, None, None, None) == 3
    assert lib.mtp_row_stats(fake, odd, 1, fake, 4, 3, 10, fake, fake, None, None) == 3
    assert lib.mtp_row_stats(fake, fake, 1, fake, 4, 3, 10, None, fake, None, None) == 1
    assert lib.mtp_tv_loss_fwd_bwd(fake, fake, 1, 1.0, 4, 3, 10, 1.0, fake, None, odd, None, None) == 3
    assert lib.mtp_tv_loss_fwd_bwd(fake, fake, 1, 1.0, 4, 3, 10, 1.0, None, None, fake, None, None) == 1
    assert lib.mtp_tv_loss_fwd_bwd(None, None, 1, 1.0, 0, 3, 10, 1.0, None, None, None, None, None) == 0
    assert lib.mtp_tv_loss_fwd_bwd(fake, fake, 5, 1.0, 4, 3, 10, 1.0, fake, None, fake, None, None) == 2


def test_query_plan_validation_without_gpu(lib):
    """Arguments are checked before any device call: ops 0-11 exist, the
    dtype must be f32 or bf16, units, gamma and V must be in range."""
    c = ctypes.c_int(0)
    r = ctypes.byref(c)
    for op in (-1, 12, 99):
        assert lib.mtp_query_plan(op, 1, 64, 3, 151936, r, r, r, r) == 1, op
    assert lib.mtp_query_plan(0, 7, 64, 3, 151936, r, r, r, r) == 2
    assert lib.mtp_query_plan(11, 1, 0, 3, 151936, r, r, r, r) == 1
    assert lib.mtp_query_plan(11, 1, 192, 0, 151936, r, r, r, r) == 1
    assert lib.mtp_query_plan(10, 1, 192, 3, 0, r, r, r, r) == 1
    assert lib.mtp_query_plan(9, 1, 64, 33, 151936, r, r, r, r) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        mtp.load_library(str(tmp_path / "missing.so"))
