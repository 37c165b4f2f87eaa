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
    for s in range(1, 7):
        assert mtp.mtp_status_string(s) not in ("ok", "unknown status")
    assert mtp.MTP_ERR_TIMEOUT == 5 and mtp.MTP_ERR_NO_DEVICE == 6
    assert "wait" in mtp.mtp_status_string(mtp.MTP_ERR_TIMEOUT)


def test_status_codes_match_header():
    """The binding's status and kernel codes are the header's enums."""
    text = open(os.path.join(ROOT, "include", "mtp_rs.h")).read()
    for name in ("MTP_OK", "MTP_ERR_INVALID_ARG", "MTP_ERR_UNSUPPORTED_DTYPE", "MTP_ERR_MISALIGNED", "MTP_ERR_CUDA",
                 "MTP_ERR_TIMEOUT", "MTP_ERR_NO_DEVICE"):
        m = re.search(rf"\b{name}\s*=\s*(\d+)", text)
        assert m and int(m.group(1)) == getattr(mtp, name), name
    for name in ("AUTO", "STREAM", "RESIDENT", "TMEM"):
        m = re.search(rf"\bMTP_KERNEL_{name}\s*=\s*(\d+)", text)
        assert m and int(m.group(1)) == getattr(mtp, "KERNEL_" + name), name
    fields = re.search(r"typedef struct mtp_tuning \{(.*?)\} mtp_tuning;", text, flags=re.S).group(1)
    fields = re.sub(r"/\*.*?\*/", "", fields, flags=re.S)
    assert tuple(re.findall(r"int (\w+);", fields)) == mtp.TUNING_FIELDS


def test_tuning_roundtrip_without_gpu(lib):
    """Kernel choices come from the explicit tuning API, never from the
    environment: set, read back, restore, and NULL clears."""
    assert all(v == 0 for v in mtp.mtp_get_tuning().values())
    with mtp.tuning(cluster_size=8, tv_kernel=mtp.KERNEL_RESIDENT, lookahead=1):
        t = mtp.mtp_get_tuning()
        assert t["cluster_size"] == 8 and t["tv_kernel"] == mtp.KERNEL_RESIDENT and t["lookahead"] == 1
        with mtp.tuning(max_clusters=3):
            assert mtp.mtp_get_tuning()["max_clusters"] == 3 and mtp.mtp_get_tuning()["cluster_size"] == 8
        assert mtp.mtp_get_tuning()["max_clusters"] == 0
    assert all(v == 0 for v in mtp.mtp_get_tuning().values())
    mtp.mtp_set_tuning(ring_slots=4)
    assert lib.mtp_set_tuning(None) == 0
    assert all(v == 0 for v in mtp.mtp_get_tuning().values())
    assert lib.mtp_get_tuning(None) == 1
    with pytest.raises(ValueError):
        mtp.mtp_set_tuning(no_such_field=1)


def test_library_reads_no_environment():
    """The product library imports no getenv: a caller's environment cannot
    change which kernel runs."""
    out = subprocess.run(["nm", "-D", "--undefined-only", mtp_build.LIB], capture_output=True, text=True).stdout
    assert "getenv" not in out
    for src in glob.glob(os.path.join(ROOT, "mtp_speculative_decoding_row_gb300", "csrc", "*")):
        assert "getenv" not in open(src).read(), src


def test_out_buffers_checked_before_launch(monkeypatch):
    """A caller-supplied result tuple of the wrong shape or dtype raises
    before the library is touched."""
    import torch

    def no_library(*a, **k):
        raise AssertionError("the library must not be called")

    monkeypatch.setattr(mtp, "load_library", no_library)
    B, g, V = 4, 3, 64
    tl = torch.zeros((B, g + 1, V))
    dl = torch.zeros((B, g, V))
    ids = torch.zeros((B, g), dtype=torch.int32)
    T = torch.ones(B)
    u = torch.zeros((B, g + 1))
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32)  # noqa: E731
    bad = mtp.VerifyResult(i32(B, g), i32(B), None, None, i32(B))  # tokens one column short
    with pytest.raises(ValueError, match="out.tokens"):
        mtp.mtp_rs_verify(tl, dl, ids, T, u, out=bad)
    bad = mtp.VerifyResult(i32(B, g + 1), torch.zeros(B), None, None, i32(B))  # float accept_len
    with pytest.raises(TypeError, match="out.accept_len"):
        mtp.mtp_rs_verify(tl, dl, ids, T, u, out=bad)
    good_no_stats = mtp.VerifyResult(i32(B, g + 1), i32(B), None, None, i32(B))
    with pytest.raises(ValueError, match="with_stats"):
        mtp.mtp_rs_verify(tl, dl, ids, T, u, with_stats=True, out=good_no_stats)
    bad = mtp.StatsResult(torch.zeros((B, g)), torch.zeros((B, g)), i32(B))  # entropy needs gamma + 1 columns
    with pytest.raises(ValueError, match="out.entropy"):
        mtp.mtp_row_stats(tl, dl, T, out=bad)
    bad = mtp.TVLossResult(torch.zeros(B), torch.zeros((B, g)), torch.zeros((B, g, V - 1)), i32(B))
    with pytest.raises(ValueError, match="out.grad"):
        mtp.mtp_tv_loss_fwd_bwd(dl, dl, out=bad)
    bad = mtp.TVLossResult(torch.zeros(B), torch.zeros((B, g)), torch.zeros((B, V, g)).transpose(1, 2), i32(B))
    with pytest.raises(ValueError, match="contiguous"):
        mtp.mtp_tv_loss_fwd_bwd(dl, dl, out=bad)
    bad = mtp.SampleResult(i32(B * g + 1), i32(B * g))
    with pytest.raises(ValueError, match="out.ids"):
        mtp.mtp_draft_sample(dl, torch.ones(B * g), torch.zeros(B * g), out=bad)


def test_check_row_flags_raises_timeout():
    import numpy as np

    mtp.check_row_flags(np.array([0, 1, 8], np.int32))
    with pytest.raises(mtp.MTPError) as e:
        mtp.check_row_flags(np.array([0, mtp.ROW_TIMEOUT], np.int32))
    assert e.value.status == mtp.MTP_ERR_TIMEOUT


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
