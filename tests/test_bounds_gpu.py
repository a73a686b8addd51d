"""The bounds-checking build (compiled with -DVARLEN_DEBUG_BOUNDS): every
plain global load and store of every kernel checks the bytes it touches
against its operand's extent and records VARLEN_ERR_DEVICE_BOUNDS instead of
accessing outside; it is the out-of-bounds check that stands in for a
sanitizer's memory check.  Ragged, padded, strided-dout,
causal, windowed, deterministic and E4M3 calls run in a child process on
that build and must report VARLEN_OK and give the normal build's results
(the same bits, except the atomic path's dQ, whose additions may come in
another order).  With the operand extents shortened by 16 bytes the
checker must fire (VARLEN_ERR_DEVICE_BOUNDS) and the context stay usable."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_build_matches_and_reports_nothing(tmp_path):
    from packed_variable_length_varlen_gb300 import build
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    from tests import bounds_cases as BC
    lib = build.build(bounds=True)
    path = str(tmp_path / "bounds.pt")
    env = dict(os.environ, VARLEN_ATTN_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "tests.bounds_cases", path], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    got = torch.load(path)
    assert got["bounds_checked"] == 1
    ref = BC.run_cases(va)
    assert ref["bounds_checked"] == 0
    for key, g in got.items():
        if not isinstance(g, dict) or key == "slack":
            continue
        assert all(s == 0 for s in g["status"]), (key, g["status"])
        for n in ("out", "lse", "dk", "dv"):
            if n in g:
                assert torch.equal(g[n], ref[key][n]), (key, n)
        if "dq" in g:
            if key.endswith("/det"):
                assert torch.equal(g["dq"], ref[key]["dq"]), key
            else:
                torch.testing.assert_close(g["dq"].float(), ref[key]["dq"].float(), rtol=2e-2, atol=1e-3)
    # the checker fires when the extents are short, and only in the checking build
    assert got["slack"]["status"] == (0, va.VARLEN_ERR_DEVICE_BOUNDS)
    assert ref["slack"]["status"] == (0, 0)
    assert got["after_slack"] == 0 and ref["after_slack"] == 0
