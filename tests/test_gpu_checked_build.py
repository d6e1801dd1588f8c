"""The access-checking build (librepops_debug.so) as a stand-in for a memory
sanitizer: its GEMM, mean + SGD and Merkle kernels test every global access
against the span of the buffer it belongs to and skip (never perform) one
outside it, reporting REPOPS_ERR_BOUNDS through the status word -- no trap,
no fault.  A set of ragged, unaligned, transposed, chained, batched and typed
workloads runs on it in a child process: no access may be reported, and
every result must equal the release library's bytes."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.slow
def test_checked_build_reports_nothing_and_matches_release(rp, tmp_path):
    from verifiable_repops_gemm_gb300 import build
    lib = build.build(checked=True)
    out = tmp_path / "checked.npz"
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_build_run.py"), lib, str(out)],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    import checked_build_run
    want = checked_build_run.workloads(rp)
    got = np.load(out)
    assert sorted(got.files) == sorted(want)
    for name, w in want.items():
        g = got[name]
        assert g.shape == w.shape, name
        assert np.array_equal(np.ascontiguousarray(g).view(np.uint8), np.ascontiguousarray(w).view(np.uint8)), name
