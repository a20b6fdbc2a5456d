"""qgemv_i4g_noalloc against the oracle and against qgemv_i4g (needs a GPU).

qgemv_i4g_noalloc serves callers that cannot hand the library a workspace:
engines whose device memory is planned once by their own allocator, and
decode loops that must not call cudaMalloc because it can wait for the whole
device.  It takes the split-reduction scratch from a fixed array inside the
library.  These shapes split the reduction, so that array is really used; two
calls in a row (different activations) check that a call does not depend on
what the previous call left in it.  A child process checks that the entry
point finds the array again after cudaDeviceReset.  This file is collected
last so that a run stopping at the first failure has already run every other
test."""
import os
import subprocess
import sys

import pytest

from gpu_util import compare, dev, host, i4g_inputs, out, par_rows, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


@pytest.mark.parametrize("O,I,S", [(3, 65536, 1), (64, 16384, 2), (100, 4096, 8)])
def test_noalloc_matches_oracle_and_workspace_entry_point(qg, O, I, S):
    gs = 64
    nws = qg.qg_workspace_bytes(qg.QG_FMT_I4G, S, I, O, gs)
    assert 0 < nws <= (4 << 20)
    _, wq, sc = i4g_inputs(O, I, S, gs, tag=O + S)
    wd, sd = dev(wq), dev(sc)
    for call in range(2):
        x, _, _ = i4g_inputs(O, I, S, gs, tag=O + S + 100 * (call + 1))
        xd = dev(x)
        ws, nws = workspace(qg, qg.QG_FMT_I4G, S, I, O, gs)
        y_ref = out(S, O)
        qg.check(qg.qgemv_i4g(y_ref, xd, wd, sd, S, I, O, gs, ws, nws))
        y = out(S, O)
        qg.check(qg.qgemv_i4g_noalloc(y, xd, wd, sd, S, I, O, gs))
        got, other = host(y, S, O), host(y_ref, S, O)
        want, mag = par_rows(orc_gemv(), O, x, wq, sc, S, I, O, gs)
        compare(got, want, mag, what=f"noalloc vs oracle, call {call + 1}")
        compare(got, other, mag, what=f"noalloc vs qgemv_i4g, call {call + 1}")
    rc, status = qg.qg_device_status()
    assert rc == qg.QG_OK and status == qg.QG_OK


def orc_gemv():
    from gpu_util import orc
    return orc().qgemv_i4g


def test_noalloc_after_device_reset():
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "noalloc_reset_child.py")
    r = subprocess.run([sys.executable, child], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok"), r.stdout
